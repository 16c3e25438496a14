// Decode kernels: fused route+attend (sekv_decode_step), list-driven attend
// (sekv_decode_attention) and the list preparation kernel it uses.
#include "decode_consumer.cuh"
#include "decode_producer.cuh"

namespace sekv {

// Routing page: lane = span.  z_h = y_h . s_S (fp32), span expands iff its
// body is non-empty and some head of the group has z_h > theta_h.  Expanded
// spans are appended, in ascending order, to this CTA's private slice of the
// entry array together with their record size prefix.
__device__ __forceinline__ void consume_route(const uint8_t* page, const PageDesc& d, int k0,
                                              const DecodeParams& P, SmemMisc* ms,
                                              float* infoc, const float* ys, size_t gs) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int kk = 32 * w + lane;
  const bool valid = kk < d.n;
  int body = 0, rank = 0;
  long long off = 0;
  float z[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) z[h] = 0.f;
  if (valid) {
    body = reinterpret_cast<const int*>(page + kAuxBody)[kk];
    rank = reinterpret_cast<const int*>(page + kAuxRank)[kk];
    off = reinterpret_cast<const long long*>(page + kAuxOff)[kk];
    const int row = kk & 63;
    const uint8_t* rbox = page + (kk >> 6) * 2 * 8192;
    const float4* y4 = reinterpret_cast<const float4*>(ys);
#pragma unroll 4
    for (int dc = 0; dc < 16; ++dc) {
      const uint8_t* box = rbox + (dc >> 3) * 8192;
      const float4 s = *reinterpret_cast<const float4*>(box + row * 128 +
                                                        (((dc & 7) ^ (row & 7)) << 4));
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h < P.G) {
          const float4 y = y4[h * 16 + dc];
          z[h] = fmaf(s.x, y.x, fmaf(s.y, y.y, fmaf(s.z, y.z, fmaf(s.w, y.w, z[h]))));
        }
      }
    }
  }
  bool hit = false;
#pragma unroll
  for (int h = 0; h < 8; ++h)
    if (h < P.G) hit |= z[h] > ms->theta[h];
  const bool ex = valid && body > 0 && hit;
  if (valid) infoc[d.a - k0 + kk] = (body > 0 && !ex) ? log2f(float(body)) : kNegInf;
  long long size = ex ? record_bytes(body, rank & 0xffff, (rank >> 16) & 0xffff) : 0;
  // inclusive warp scan of sizes
  long long incl = size;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const uint32_t bal = __ballot_sync(0xffffffffu, ex);
  if (lane == 31) ms->wbytes[w] = incl;
  if (lane == 0) ms->wcnt[w] = __popc(bal);
  named_bar(1, kConsumers);
  int base_n = ms->n_local;
  long long base_b = ms->bytes_local;
  for (int ww = 0; ww < w; ++ww) {
    base_n += ms->wcnt[ww];
    base_b += ms->wbytes[ww];
  }
  if (ex) {
    const int pos = base_n + __popc(bal & ((1u << lane) - 1u));
    const long long cum = base_b + incl - size;
    int4* dst = reinterpret_cast<int4*>(P.entries + gs + k0 + pos);
    dst[0] = make_int4(d.a + kk, body, rank, 0);
    dst[1] = make_int4(int(uint32_t(off)), int(off >> 32), int(uint32_t(cum)), int(cum >> 32));
  }
  named_bar(1, kConsumers);
  if (tid == 0) {
    int tn = 0;
    long long tb = 0;
    for (int ww = 0; ww < kConsumerWarps; ++ww) {
      tn += ms->wcnt[ww];
      tb += ms->wbytes[ww];
    }
    ms->n_local += tn;
    ms->bytes_local += tb;
  }
}

__device__ void consumer_warps(uint8_t* smem, SmemMisc* ms, const DecodeParams& P, int g, int j,
                               int b, int c) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int G = P.G;
  const int n_sp = P.n_spans[b];
  const int n_full = P.n_sink + n_sp + P.n_recent;
  int f0, f1, k0, k1;
  fixed_range(j, P.cg, n_full, n_sp, P.fused, f0, f1, k0, k1);
  const size_t gs = size_t(g) * P.max_spans;
  float* infoc = reinterpret_cast<float*>(smem + kOffInfo);  // summary bias per span
  float* qs = reinterpret_cast<float*>(smem + kOffScratch);         // prologue only
  float* ys = reinterpret_cast<float*>(smem + kOffScratch + 4096);  // routing pages only

  pdl_wait();
  WarpAcc A;
  const __nv_bfloat16* qg = P.q + (size_t(b) * P.Hq + size_t(c) * G) * kHeadDim;
  {
    const int r0 = lane >> 2;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int k = 16 * s + 2 * (lane & 3);
      A.qa[s][0] = r0 < G ? *reinterpret_cast<const uint32_t*>(qg + r0 * kHeadDim + k) : 0u;
      A.qa[s][1] = r0 < G ? *reinterpret_cast<const uint32_t*>(qg + r0 * kHeadDim + k + 8) : 0u;
    }
  }
#pragma unroll
  for (int t = 0; t < 16; ++t) A.o[t][0] = A.o[t][1] = 0.f;
  A.m_row = kNegInf;
  A.l_part = 0.f;
  ExpAcc X;
  X.had = false;

  if (P.fused) {
    for (int i = tid; i < 8 * kHeadDim; i += kConsumers)
      qs[i] = (i / kHeadDim) < G ? __bfloat162float(qg[i]) : 0.f;
    if (tid < 8) ms->theta[tid] = tid < G ? P.theta[c * G + tid] : 0.f;
    named_bar(1, kConsumers);
    // y_h = W_r[c] q_h from the staged rows (padded stride: conflict-free
    // 16-byte loads), one routing coordinate per thread, heads hh, hh+2, ...
    if (!mbar_wait(&ms->wr_bar, 0, kWaitLimit) && tid == 0)
      set_device_error(P.status, DEV_WAIT_TIMEOUT, 5);
    const int jr = tid & 63, hh = tid >> 6;
    const float4* wrow = reinterpret_cast<const float4*>(smem + kOffWr + jr * kWrStride);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int d4 = 0; d4 < 32; ++d4) {
      const float4 wv = wrow[d4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (hh + 2 * i < G) {
          const float4 qv = reinterpret_cast<const float4*>(qs + (hh + 2 * i) * kHeadDim)[d4];
          acc[i] = fmaf(wv.x, qv.x, fmaf(wv.y, qv.y, fmaf(wv.z, qv.z, fmaf(wv.w, qv.w, acc[i]))));
        }
      }
    }
    named_bar(1, kConsumers);  // qs is dead; ys may overwrite nothing it needs
#pragma unroll
    for (int i = 0; i < 4; ++i) ys[(hh + 2 * i) * kRouteDim + jr] = acc[i];
    named_bar(1, kConsumers);
  }

  int slot = 0;
  uint32_t phase = 0;
  for (;;) {
    if (!mbar_wait(&ms->full[slot], phase, kWaitLimit)) {
      if (tid == 0) set_device_error(P.status, DEV_WAIT_TIMEOUT, 4);
      break;
    }
    const PageDesc d = ms->desc[slot];
    const uint8_t* page = smem + slot * kPageStride;
    const uint32_t pu = smem_u32(page);
    switch (d.type) {
      case PG_ROUTE:
        consume_route(page, d, k0, P, ms, infoc, ys, gs);
        if (d.flag) {
          __threadfence();
          named_bar(1, kConsumers);
          if (tid == 0) {
            P.cta_n[size_t(g) * P.cg + j] = ms->n_local;
            P.cta_bytes[size_t(g) * P.cg + j] = ms->bytes_local;
            __threadfence();
            atomicAdd(&P.groups[g].published, 1);
          }
        }
        break;
      case PG_INFO: {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(page);
        for (int i = tid; i < d.n; i += kConsumers) {
          const int inf = src[i], body = inf & 0x7fff;
          infoc[i] = (body > 0 && !(inf & 0x8000)) ? log2f(float(body)) : kNegInf;
        }
        named_bar(1, kConsumers);
        break;
      }
      case PG_FULL:
        consume_kv_tile(A, pu, pu + 16384, d.n, nullptr, P.scale_log2);
        break;
      case PG_SUM:
        consume_kv_tile(A, pu, pu + 16384, d.n, infoc + (d.a - k0), P.scale_log2);
        break;
      case PG_EXP:  // one large record, split over pages; all warps share its tokens
        if (d.off_a >= 0) exp_key(A, X, page + d.off_a, d.rk, P.scale_log2);
        if (d.n > 0)
          exp_tokens(A, X, page + d.off_uk, page + d.off_uv, d.n, d.rk, d.rv, 16 * w,
                     16 * kConsumerWarps);
        if (d.off_b >= 0) exp_value(A, X, page + d.off_b, d.rv);
        break;
      case PG_EXPM:  // several small records: warp w takes records w, w+4, ...
        for (int i = w; i < d.n; i += kConsumerWarps) {
          const RecInfo ri = ms->rec[slot][i];
          const uint8_t* part = page + ri.off;
          const RecordLayout RL = record_layout(ri.b, ri.rk, ri.rv);
          exp_key(A, X, part, ri.rk, P.scale_log2);
          exp_tokens(A, X, part + RL.uk, part + RL.uv, ri.b, ri.rk, ri.rv, 0, 16);
          exp_value(A, X, part + RL.vpart, ri.rv);
        }
        break;
      default:
        break;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->empty[slot]);
    if (d.type == PG_END) break;
    if (++slot == kPages) {
      slot = 0;
      phase ^= 1u;
    }
  }

  // ---- merge the four warps' states into this CTA's partial --------------
  named_bar(1, kConsumers);  // every warp is past its last page
  Partial* wp = reinterpret_cast<Partial*>(smem);  // pages are free now
  {
    const int r0 = lane >> 2;
    float l_row = A.l_part + __shfl_xor_sync(0xffffffffu, A.l_part, 1);
    l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
    if (r0 < G) {
      if ((lane & 3) == 0) {
        wp[w].m[r0] = A.m_row;
        wp[w].l[r0] = l_row;
      }
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        wp[w].o[r0][8 * t + 2 * (lane & 3)] = A.o[t][0];
        wp[w].o[r0][8 * t + 2 * (lane & 3) + 1] = A.o[t][1];
      }
    }
  }
  named_bar(1, kConsumers);
  Partial* mine = P.partials + size_t(g) * P.cg + j;
  for (int h = 0; h < G; ++h) {
    float M = kNegInf;
#pragma unroll
    for (int ww = 0; ww < kConsumerWarps; ++ww) M = fmaxf(M, wp[ww].m[h]);
    float L = 0.f, O = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int ww = 0; ww < kConsumerWarps; ++ww) {
        const float sc = exp2f(wp[ww].m[h] - M);
        L = fmaf(wp[ww].l[h], sc, L);
        O = fmaf(wp[ww].o[h][tid], sc, O);
      }
    }
    mine->o[h][tid] = O;
    if (tid == 0) {
      mine->m[h] = M;
      mine->l[h] = L;
    }
  }
  __threadfence();
  named_bar(1, kConsumers);
  if (tid == 0) {
    const int old = atomicAdd(&P.groups[g].done, 1);
    ms->is_last = (old == P.cg - 1);
  }
  named_bar(1, kConsumers);
  if (!ms->is_last) return;

  // ---- last CTA of this KV head: merge the partials, write the output -----
  __threadfence();
  const int cg = P.cg;
  const Partial* parts = P.partials + size_t(g) * cg;
  float* sm_m = reinterpret_cast<float*>(smem + 32768);   // [cg][8]
  float* sm_s = sm_m + kMaxCgSmem * 8;                    // [cg][8] scales
  float* sm_l = sm_s + kMaxCgSmem * 8;                    // [cg][8]
  float* sm_ML = sm_l + kMaxCgSmem * 8;                   // M[8], L[8]
  for (int i = tid; i < cg * 8; i += kConsumers) {
    const int jj = i >> 3, h = i & 7;
    sm_m[i] = h < G ? __ldcg(&parts[jj].m[h]) : kNegInf;
    sm_l[i] = h < G ? __ldcg(&parts[jj].l[h]) : 0.f;
  }
  named_bar(1, kConsumers);
  if (tid < G) {
    float M = kNegInf;
    for (int jj = 0; jj < cg; ++jj) M = fmaxf(M, sm_m[jj * 8 + tid]);
    float L = 0.f;
    if (M != kNegInf)
      for (int jj = 0; jj < cg; ++jj) L = fmaf(sm_l[jj * 8 + tid], exp2f(sm_m[jj * 8 + tid] - M), L);
    sm_ML[tid] = M;
    sm_ML[8 + tid] = L;
  }
  named_bar(1, kConsumers);
  for (int i = tid; i < cg * 8; i += kConsumers) {
    const int h = i & 7;
    const float M = h < G ? sm_ML[h] : kNegInf;
    sm_s[i] = (M == kNegInf) ? 0.f : exp2f(sm_m[i] - M);
  }
  named_bar(1, kConsumers);
  for (int h = 0; h < G; ++h) {
    float Oa[4] = {0.f, 0.f, 0.f, 0.f};
    int jj = 0;
    for (; jj + 4 <= cg; jj += 4) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcg(&parts[jj + u].o[h][tid]);
#pragma unroll
      for (int u = 0; u < 4; ++u) Oa[u] = fmaf(v[u], sm_s[(jj + u) * 8 + h], Oa[u]);
    }
    for (; jj < cg; ++jj) Oa[0] = fmaf(__ldcg(&parts[jj].o[h][tid]), sm_s[jj * 8 + h], Oa[0]);
    const float O = (Oa[0] + Oa[1]) + (Oa[2] + Oa[3]);
    const float L = sm_ML[8 + h];
    const size_t row = size_t(b) * P.Hq + size_t(c) * G + h;
    P.out[row * kHeadDim + tid] = L > 0.f ? O / L : 0.f;
    if (tid == 0 && P.lse != nullptr)
      P.lse[row] = L > 0.f ? (sm_ML[h] + log2f(L)) * kLn2 : kNegInf;
  }
  if (P.expanded_out != nullptr && P.fused) {
    // concatenate the CTAs' ascending slices
    int* pre = reinterpret_cast<int*>(sm_ML + 16);
    if (tid == 0) {
      int acc = 0;
      for (int jj = 0; jj < cg; ++jj) {
        pre[jj] = acc;
        acc += __ldcg(P.cta_n + size_t(g) * cg + jj);
      }
      pre[cg] = acc;
    }
    named_bar(1, kConsumers);
    for (int jj = 0; jj < cg; ++jj) {
      int a0, a1, sk0, a2;
      fixed_range(jj, cg, n_full, n_sp, 1, a0, a1, sk0, a2);
      const int cnt = pre[jj + 1] - pre[jj];
      for (int i = tid; i < cnt; i += kConsumers)
        P.expanded_out[gs + pre[jj] + i] = __ldcg(&P.entries[gs + sk0 + i].k);
    }
    if (tid == 0 && P.n_expanded_out != nullptr) P.n_expanded_out[g] = pre[cg];
  }
  named_bar(1, kConsumers);
  if (tid == 0) {
    P.groups[g].published = 0;
    P.groups[g].done = 0;
  }
}

// grid: (cg, Hkv, B); block: 4 consumer warps + 1 producer warp
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  SmemMisc* ms = reinterpret_cast<SmemMisc*>(smem + kOffMisc);
  const int j = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int g = b * P.Hkv + c;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPages; ++s) {
      mbar_init(&ms->full[s], 1);
      mbar_init(&ms->empty[s], kConsumerWarps);
    }
    mbar_init(&ms->wr_bar, 1);
    ms->n_local = 0;
    ms->bytes_local = 0;
    ms->is_last = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (threadIdx.x >= kConsumers)
    producer_warp(smem, ms, P, g, j, b, c);
  else
    consumer_warps(smem, ms, P, g, j, b, c);
}

// ----------------------------------------------------------------------------
// list mode: span info and expansion entries from a caller's ascending list
// ----------------------------------------------------------------------------


__global__ void __launch_bounds__(256) prep_list_kernel(const PrepParams P) {
  __shared__ long long scan[256];
  __shared__ long long carry;
  const int g = blockIdx.x, b = g / P.Hkv, tid = threadIdx.x;
  const size_t gs = size_t(g) * P.max_spans;
  const int n_sp = P.n_spans[b];
  int ne = P.n_expanded[g];
  if (ne < 0 || ne > n_sp) {
    if (tid == 0) set_device_error(P.status, DEV_BAD_LIST, g);
    ne = 0;
  }
  for (int k = tid; k < n_sp; k += 256)
    P.info[gs + k] = uint16_t(P.body_len[size_t(b) * P.max_spans + k] & 0x7fff);
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int e0 = 0; e0 < ne; e0 += 256) {
    const int e = e0 + tid;
    long long size = 0;
    int k = -1, body = 0, rank = 0;
    if (e < ne) {
      k = P.expanded[gs + e];
      const int prev = e > 0 ? P.expanded[gs + e - 1] : -1;
      bool okk = k >= 0 && k < n_sp && k > prev;
      if (okk) {
        body = P.body_len[size_t(b) * P.max_spans + k];
        rank = P.rec_rank[gs + k];
        okk = body > 0 && (rank & 0xffff) <= SEKV_MAX_RANK && ((rank >> 16) & 0xffff) <= SEKV_MAX_RANK;
      }
      if (!okk) {
        set_device_error(P.status, DEV_BAD_LIST, e);
        body = 0;
      } else {
        size = record_bytes(body, rank & 0xffff, (rank >> 16) & 0xffff);
      }
    }
    scan[tid] = size;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {
      const long long v = tid >= o ? scan[tid - o] : 0;
      __syncthreads();
      scan[tid] += v;
      __syncthreads();
    }
    const long long cum = carry + scan[tid] - size;
    if (e < ne) {
      const long long off = body > 0 ? (P.staged_off ? P.staged_off[gs + e] : P.rec_off[gs + k]) : 0;
      int4* dst = reinterpret_cast<int4*>(P.entries + gs + e);
      dst[0] = make_int4(k, body, rank, 0);
      dst[1] = make_int4(int(uint32_t(off)), int(off >> 32), int(uint32_t(cum)), int(cum >> 32));
      if (body > 0) P.info[gs + k] = uint16_t((body & 0x7fff) | 0x8000);
    }
    __syncthreads();
    if (tid == 255) carry += scan[255];
    __syncthreads();
  }
  for (int jj = tid; jj < P.cg; jj += 256) {
    P.cta_n[size_t(g) * P.cg + jj] = jj == 0 ? ne : 0;
    P.cta_bytes[size_t(g) * P.cg + jj] = jj == 0 ? carry : 0;
  }
  if (tid == 0) P.groups[g].published = P.cg;
}

}  // namespace sekv
