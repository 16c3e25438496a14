// Prefill build kernels: segmentation, planning, anchor gather, summaries.
// (The batched span SVD is in build_svd.cu.)
#include "build.cuh"

namespace sekv {

// ----------------------------------------------------------------------------
// segmentation: one CTA per sequence.  Candidates (H_t > tau, float32, strict)
// go into a shared bitmask; one thread walks the span chain:
//   next(s) = min(first candidate t >= s + len_min, s + len_max),
// the last span ends at the end of the middle region [n_sink, T - n_recent).
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) seg_kernel(const BuildParams P) {
  extern __shared__ uint32_t bits[];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int m0 = P.n_sink, m1 = P.T - P.n_recent;
  const int n_mid = m1 > m0 ? m1 - m0 : 0;
  const int words = (n_mid + 31) / 32;
  if (b == 0 && tid < 16) P.counters[tid] = 0;  // class counts/cursors for this call
  const float* Hb = P.H + size_t(b) * P.T;
  for (int w = wid; w < words; w += blockDim.x / 32) {
    const int t = m0 + 32 * w + lane;
    const bool cand = t < m1 && Hb[t] > P.tau;
    const uint32_t word = __ballot_sync(0xffffffffu, cand);
    if (lane == 0) bits[w] = word;
  }
  __syncthreads();
  if (tid != 0) return;
  int32_t* starts = P.starts + size_t(b) * P.max_spans;
  int32_t* body = P.body_len + size_t(b) * P.max_spans;
  int k = 0, s = m0;
  while (s < m1) {
    if (k >= P.max_spans) {
      set_device_error(P.status, DEV_BAD_LIST, b);  // more spans than max_spans
      break;
    }
    // first candidate in [s + len_min, min(s + len_max, m1))
    const int lo = s + P.len_min, hi = min(s + P.len_max, m1);
    int next = s + P.len_max;
    for (int t = lo; t < hi;) {
      const int rel = t - m0;
      uint32_t word = bits[rel >> 5] >> (rel & 31);
      if (word) {
        const int c = t + __ffs(word) - 1;
        if (c < hi) next = c;
        break;
      }
      t += 32 - (rel & 31);
    }
    if (next > m1) next = m1;
    starts[k] = s;
    body[k] = next - s - 1;
    ++k;
    s = next;
  }
  P.n_spans[b] = k;
  for (int kk = k; kk < P.max_spans; ++kk) body[kk] = 0;
}

// ----------------------------------------------------------------------------
// planning: one CTA per (sequence, KV head).  Ranks from the soft gates
// (longest prefix with g > 0.5, at most min(rank_cap, b) components), record
// sizes and offsets inside the group, SVD work lists by size class.  The last
// CTA turns the group totals into group base offsets in the store.
// ----------------------------------------------------------------------------
__device__ __forceinline__ int gate_rank(const float* g, int R) {
  int r = 0;
  while (r < R && g[r] > 0.5f) ++r;
  return r;
}

__global__ void __launch_bounds__(256) plan_kernel(const BuildParams P) {
  __shared__ long long scan[256];
  __shared__ long long carry;
  __shared__ int ccount[kSvdClasses], cbase[kSvdClasses];
  __shared__ int is_last;
  const int g = blockIdx.x, b = g / P.Hkv, c = g % P.Hkv, tid = threadIdx.x;
  const int n_sp = P.n_spans[b];
  const size_t gs = size_t(g) * P.max_spans;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int k0 = 0; k0 < P.max_spans; k0 += 256) {
    const int k = k0 + tid;
    long long size = 0;
    int cls = -1, rk = 0, rv = 0;
    if (k < n_sp) {
      const int bl = P.body_len[size_t(b) * P.max_spans + k];
      if (bl > 0) {
        const int R = bl < P.rank_cap ? bl : P.rank_cap;
        const float* gk = P.gates + ((size_t(b) * P.Hkv + c) * 2 * P.max_spans + k) * P.rank_cap;
        const float* gv = gk + size_t(P.max_spans) * P.rank_cap;
        rk = gate_rank(gk, R);
        rv = gate_rank(gv, R);
        size = record_bytes(bl, rk, rv);
        cls = bl <= 32 ? 0 : bl <= 64 ? 1 : bl <= 128 ? 2 : 3;
      }
    }
    if (k < P.max_spans) P.rec_rank[gs + k] = rk | (rv << 16);
    if (tid < kSvdClasses) ccount[tid] = 0;
    scan[tid] = size;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {
      const long long v = tid >= o ? scan[tid - o] : 0;
      __syncthreads();
      scan[tid] += v;
      __syncthreads();
    }
    if (k < P.max_spans) P.rel_off[gs + k] = carry + scan[tid] - size;
    int slot = -1;
    if (cls >= 0) slot = atomicAdd(&ccount[cls], 2);  // key and value items
    __syncthreads();
    if (tid < kSvdClasses) cbase[tid] = ccount[tid] ? atomicAdd(&P.counters[tid], ccount[tid]) : 0;
    __syncthreads();
    if (cls >= 0) {
      const int pos = cbase[cls] + slot;
      if (pos + 1 < P.cls_cap) {
        int32_t* lst = P.cls_list + size_t(cls) * P.cls_cap;
        lst[pos] = int32_t((gs + k) * 2);
        lst[pos + 1] = int32_t((gs + k) * 2 + 1);
      }
    }
    __syncthreads();
    if (tid == 0) carry += scan[255];
    __syncthreads();
  }
  if (tid == 0) {
    P.gtotal[g] = carry;
    __threadfence();
    is_last = atomicAdd(&P.counters[8], 1) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last || tid != 0) return;
  __threadfence();
  long long acc = 0;
  for (int gg = 0; gg < gridDim.x; ++gg) {
    P.gbase[gg] = acc;
    acc += __ldcg(reinterpret_cast<const long long*>(P.gtotal) + gg);
  }
  if (acc > P.store_capacity) set_device_error(P.status, DEV_STAGING_FULL, int(acc >> 20));
  P.counters[8] = 0;
}

// ----------------------------------------------------------------------------
// full-resolution rows: sinks, one anchor per span, recent window; rows past
// them (up to the capacity) are zeroed.  grid (B*Hkv, 32), 256 threads, 16 B
// per thread per step.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gather_kernel(const BuildParams P) {
  const int g = blockIdx.x, b = g / P.Hkv, part = blockIdx.y, tid = threadIdx.x;
  const int n_sp = P.n_spans[b];
  const int cap = P.n_sink + P.max_spans + P.n_recent;
  const int n_full = P.n_sink + n_sp + P.n_recent;
  const int4* Ksrc = reinterpret_cast<const int4*>(P.K + size_t(g) * P.T * kHeadDim);
  const int4* Vsrc = reinterpret_cast<const int4*>(P.V + size_t(g) * P.T * kHeadDim);
  int4* Kd = reinterpret_cast<int4*>(P.k_full + size_t(g) * cap * kHeadDim);
  int4* Vd = reinterpret_cast<int4*>(P.v_full + size_t(g) * cap * kHeadDim);
  const int32_t* starts = P.starts + size_t(b) * P.max_spans;
  const int per_row = kHeadDim * 2 / 16;  // 16 int4 per row
  for (int idx = part * 256 + tid; idx < cap * per_row; idx += gridDim.y * 256) {
    const int row = idx / per_row, col = idx % per_row;
    int4 kv = make_int4(0, 0, 0, 0), vv = kv;
    if (row < n_full) {
      int t;
      if (row < P.n_sink) t = row;
      else if (row < P.n_sink + n_sp) t = starts[row - P.n_sink];
      else t = P.T - P.n_recent + (row - P.n_sink - n_sp);
      kv = Ksrc[size_t(t) * per_row + col];
      vv = Vsrc[size_t(t) * per_row + col];
    }
    Kd[idx] = kv;
    Vd[idx] = vv;
  }
}

// ----------------------------------------------------------------------------
// summaries: one warp per (group, span).  Lane l owns dims 4l..4l+3.
//   kbar, vbar = uniform means of the body rows (bf16, round to nearest even)
//   s = u / |u|, u = W_r (sum_i H_i k_i)  (= sum_i H_i W_r k_i)
// grid (ceil(max_spans / 8), B*Hkv), 256 threads
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) summary_kernel(const BuildParams P) {
  __shared__ float kh[8][kHeadDim];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y, b = g / P.Hkv, c = g % P.Hkv;
  // decode-time maintenance: spans only_k[b] .. only_k[b] + only_n[b] - 1
  const int j = blockIdx.x * 8 + wid;
  const int k = P.only_k != nullptr ? (j < P.only_n[b] ? P.only_k[b] + j : -1) : j;
  const size_t gs = size_t(g) * P.max_spans;
  if (k < 0 || k >= P.max_spans) return;
  const int n_sp = P.only_k != nullptr ? k + 1 : P.n_spans[b];
  const int bl = k < n_sp ? P.body_len[size_t(b) * P.max_spans + k] : 0;
  float4 ks = make_float4(0.f, 0.f, 0.f, 0.f), vs = ks, hs = ks;
  if (bl > 0) {
    const int t0 = P.starts[size_t(b) * P.max_spans + k] + 1;
    const float* Hb = P.H + size_t(b) * P.T;
    const uint2* Kr = reinterpret_cast<const uint2*>(P.K + (size_t(g) * P.T + t0) * kHeadDim) + lane;
    const uint2* Vr = reinterpret_cast<const uint2*>(P.V + (size_t(g) * P.T + t0) * kHeadDim) + lane;
    for (int i = 0; i < bl; ++i) {
      const uint2 kw = Kr[size_t(i) * 32], vw = Vr[size_t(i) * 32];
      const float h = Hb[t0 + i];
      const __nv_bfloat162 k01 = *reinterpret_cast<const __nv_bfloat162*>(&kw.x);
      const __nv_bfloat162 k23 = *reinterpret_cast<const __nv_bfloat162*>(&kw.y);
      const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162*>(&vw.x);
      const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162*>(&vw.y);
      const float2 a = __bfloat1622float2(k01), bb = __bfloat1622float2(k23);
      const float2 va = __bfloat1622float2(v01), vb = __bfloat1622float2(v23);
      ks.x += a.x; ks.y += a.y; ks.z += bb.x; ks.w += bb.y;
      vs.x += va.x; vs.y += va.y; vs.z += vb.x; vs.w += vb.y;
      hs.x = fmaf(h, a.x, hs.x); hs.y = fmaf(h, a.y, hs.y);
      hs.z = fmaf(h, bb.x, hs.z); hs.w = fmaf(h, bb.y, hs.w);
    }
  }
  const float inv = bl > 0 ? 1.f / float(bl) : 0.f;
  __nv_bfloat162 o01 = __floats2bfloat162_rn(ks.x * inv, ks.y * inv);
  __nv_bfloat162 o23 = __floats2bfloat162_rn(ks.z * inv, ks.w * inv);
  uint2 ow;
  ow.x = *reinterpret_cast<uint32_t*>(&o01);
  ow.y = *reinterpret_cast<uint32_t*>(&o23);
  reinterpret_cast<uint2*>(P.k_sum + (gs + k) * kHeadDim)[lane] = ow;
  o01 = __floats2bfloat162_rn(vs.x * inv, vs.y * inv);
  o23 = __floats2bfloat162_rn(vs.z * inv, vs.w * inv);
  ow.x = *reinterpret_cast<uint32_t*>(&o01);
  ow.y = *reinterpret_cast<uint32_t*>(&o23);
  reinterpret_cast<uint2*>(P.v_sum + (gs + k) * kHeadDim)[lane] = ow;
  kh[wid][4 * lane + 0] = hs.x;
  kh[wid][4 * lane + 1] = hs.y;
  kh[wid][4 * lane + 2] = hs.z;
  kh[wid][4 * lane + 3] = hs.w;
  __syncwarp();
  float u[2] = {0.f, 0.f};
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const float4* wrow =
        reinterpret_cast<const float4*>(P.W_r + (size_t(c) * kRouteDim + lane + 32 * jj) * kHeadDim);
    float acc = 0.f;
    for (int d4 = 0; d4 < 32; ++d4) {
      const float4 w = __ldg(wrow + d4);
      acc = fmaf(w.x, kh[wid][4 * d4], fmaf(w.y, kh[wid][4 * d4 + 1],
                 fmaf(w.z, kh[wid][4 * d4 + 2], fmaf(w.w, kh[wid][4 * d4 + 3], acc))));
    }
    u[jj] = acc;
  }
  float n2 = u[0] * u[0] + u[1] * u[1];
#pragma unroll
  for (int o = 16; o; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
  const float sc = (bl > 0 && n2 > 0.f) ? rsqrtf(n2) : 0.f;
  float* srow = P.s_route + (gs + k) * kRouteDim;
  srow[lane] = u[0] * sc;
  srow[lane + 32] = u[1] * sc;
}

}  // namespace sekv
