// The decode kernel's body, a template on KS (rank k-steps of 16: ranks up
// to 16 KS).  Each KS is instantiated in a translation unit of its own.
//
// Per warp: an arena of kArenaGran granules used as a ring (items are placed
// contiguously, wrapping to the arena start when one does not fit at the
// end), up to kMaxItems items in flight, each with its own mbarrier.  The
// warp issues and consumes its items itself, in order, so no handover
// between warps is needed; the only CTA-wide synchronisation is the routing
// barrier (every span of the CTA routed, the record list final) and the
// merge at the end.
#pragma once

#include "decode_consumer.cuh"

namespace sekv {

constexpr unsigned kFull = 0xffffffffu;

// Everything a CTA derives from its block index (uniform over the CTA).
struct Ctx {
  int g, j, b, c;
  int f0, f1, k0, k1;
  int nfp;      // full-resolution pages
  int n_fixed;  // full-resolution pages + summary pages
  int n_rp;     // routing pages (fused mode)
  size_t gs;    // g * max_spans
  size_t bs;    // b * max_spans
};

// Issue state of one warp (every lane holds the same values).
struct WarpQ {
  int head, tail;   // arena granule counters (monotone)
  int ni, nd;       // items issued / consumed
  int pk;           // pending claim: 0 none, 1 fixed page, 2 record
  int pidx;         // its index (fixed page, or record entry)
  int ppart, pnp;   // record: next part, parts
  int fixed_out;    // fixed-page queue exhausted
  int rec_out;      // record queue exhausted
  int ok;           // no wait has run out
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Place an item of `bytes` in warp w's arena: returns the granule counter of
// its start, or -1 if it does not fit yet.  An empty arena starts over at
// its beginning, so that every item up to the arena's size fits eventually.
__device__ __forceinline__ int arena_place(WarpQ& Q, uint32_t bytes) {
  const int gsz = int((bytes + kGran - 1) / kGran);
  if (Q.head == Q.tail) {
    Q.head = Q.tail = (Q.head + kArenaGran - 1) / kArenaGran * kArenaGran;
  }
  int start = Q.head;
  const int pos = start % kArenaGran;
  if (pos + gsz > kArenaGran) start += kArenaGran - pos;
  if (start + gsz - Q.tail > kArenaGran) return -1;
  return start;
}

// Arm item `it` (lane 0): descriptor, then the barrier with its bytes, then
// its copies.  The descriptor is published by the barrier's phase
// completion, which the consuming lanes acquire when they wait on it.
__device__ __forceinline__ void arm_item(SmemMisc* ms, int w, int slot, const Item& it,
                                         uint32_t bytes) {
  ms->desc[w][slot] = it;
  // the warp's earlier reads of this arena space (generic proxy) come
  // before the copies that overwrite it (async proxy)
  fence_proxy_async_smem();
  mbar_arrive_expect_tx(&ms->bar[w][slot], bytes);
}

// Issue the warp's next items while it has room: first any claim still
// pending, then new claims, records before fixed pages once routing is done.
static __device__ __noinline__ void issue_more(uint8_t* smem, SmemMisc* ms, const DecodeParams& P,
                                        const Ctx& C, WarpQ& Q, bool routed) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const RecEntry* ents = reinterpret_cast<const RecEntry*>(smem + kOffEntries);
  while (Q.ok && Q.ni - Q.nd < kMaxItems) {
    if (Q.pk == 0 && routed && !Q.rec_out) {
      int e = 0;
      if (lane == 0) e = atomicAdd(&ms->rec_next, 1);
      e = __shfl_sync(kFull, e, 0);
      if (e < ms->n_rec) {
        const RecEntry en = ents[e];
        const int rK = en.rank & 0xffff, rV = (en.rank >> 16) & 0xffff;
        if (rK > P.rank_lim || rV > P.rank_lim) {
          if (lane == 0) set_device_error(P.status, DEV_BAD_RANK, rK > rV ? rK : rV);
          continue;  // skipped
        }
        Q.pk = 2;
        Q.pidx = e;
        Q.ppart = 0;
        Q.pnp = record_parts(en.body, rK, rV);
      } else {
        Q.rec_out = 1;
      }
    }
    if (Q.pk == 0 && !Q.fixed_out) {
      int f = 0;
      if (lane == 0) f = atomicAdd(&ms->fixed_next, 1);
      f = __shfl_sync(kFull, f, 0);
      if (f < C.n_fixed) {
        Q.pk = 1;
        Q.pidx = f;
      } else {
        Q.fixed_out = 1;
      }
    }
    if (Q.pk == 0) break;

    Item it{};
    uint32_t bytes = 0;
    int64_t s0 = 0, s1 = 0;
    uint32_t n0 = 0, n1 = 0;
    int64_t roff = 0;
    if (Q.pk == 1) {
      const bool full = Q.pidx < C.nfp;
      it.type = full ? IT_FULL : IT_SUM;
      it.a = full ? C.f0 + kRows * Q.pidx : C.k0 + kRows * (Q.pidx - C.nfp);
      const int e = full ? C.f1 : C.k1;
      it.n = (e - it.a) < kRows ? (e - it.a) : kRows;
      bytes = kRowPageBytes;
    } else {
      const RecEntry en = ents[Q.pidx];
      const int b = en.body, rK = en.rank & 0xffff, rV = (en.rank >> 16) & 0xffff;
      const RecordLayout L = record_layout(b, rK, rV);
      roff = (int64_t(uint32_t(en.off_lo)) | (int64_t(en.off_hi) << 32));
      it.rk = rK;
      it.rv = rV;
      if (Q.pnp == 1) {
        it.type = IT_REC;
        it.n = b;
        n0 = uint32_t(L.total);
      } else if (Q.ppart == 0) {
        it.type = IT_KEY;
        n0 = uint32_t(L.uk);
      } else if (Q.ppart < Q.pnp - 1) {
        const int rows = split_rows(rK, rV);
        const int i0 = (Q.ppart - 1) * rows;
        it.type = IT_UT;
        it.a = i0;
        it.n = (b - i0) < rows ? (b - i0) : rows;
        it.uv = 2 * it.n * r8(rK);
        s0 = L.uk + 2 * int64_t(i0) * r8(rK);
        n0 = uint32_t(it.uv);
        s1 = L.uv + 2 * int64_t(i0) * r8(rV);
        n1 = uint32_t(2 * it.n * r8(rV));
      } else {
        it.type = IT_VAL;
        s0 = L.vpart;
        n0 = uint32_t(L.total - L.vpart);
      }
      bytes = n0 + n1;
    }
    const int start = arena_place(Q, bytes);
    if (start < 0) break;  // the claim stays pending until space frees
    const int slot = Q.ni % kMaxItems;
    const int gsz = int((bytes + kGran - 1) / kGran);
    it.boff = kOffArena + w * kArenaBytes + (start % kArenaGran) * kGran;
    it.end = start + gsz;
    if (lane == 0) {
      arm_item(ms, w, slot, it, bytes);
      uint8_t* dst = smem + it.boff;
      uint64_t* bar = &ms->bar[w][slot];
      const uint64_t pol = policy_evict_first();
      if (Q.pk == 1) {
        const bool full = it.type == IT_FULL;
        tma_g2s_4d_hint(dst, full ? &P.tm_kfull : &P.tm_ksum, 0, it.a, 0, C.g, bar, pol);
        tma_g2s_4d_hint(dst + 2 * kRowHalf, full ? &P.tm_vfull : &P.tm_vsum, 0, it.a, 0, C.g,
                        bar, pol);
      } else {
        const uint8_t* rec = P.store + roff;
        if (n0) bulk_g2s_hint(dst, rec + s0, n0, bar, pol);
        if (n1) bulk_g2s_hint(dst + n0, rec + s1, n1, bar, pol);
      }
    }
    Q.head = it.end;
    ++Q.ni;
    if (Q.pk == 1 || ++Q.ppart == Q.pnp) Q.pk = 0;
  }
}

// Wait (parked, bounded) for the warp's next item; false if the wait ran out.
__device__ __forceinline__ bool wait_item(SmemMisc* ms, const WarpQ& Q) {
  const int w = threadIdx.x >> 5;
  return mbar_wait_parked(&ms->bar[w][Q.nd % kMaxItems], uint32_t((Q.nd / kMaxItems) & 1));
}

// Consume the warp's next (landed) item.
template <int KS>
__device__ __forceinline__ void consume_item(const uint8_t* smem, SmemMisc* ms, const Ctx& C,
                                             const DecodeParams& P, WarpQ& Q, WarpAcc& A,
                                             ExpAcc<KS>& X) {
  const int w = threadIdx.x >> 5;
  const Item it = ms->desc[w][Q.nd % kMaxItems];
  const uint8_t* base = smem + it.boff;
  const uint32_t bu = smem_u32(base);
  const float* bias = reinterpret_cast<const float*>(smem + kOffBias);
  if (it.type == IT_FULL || it.type == IT_SUM) {
    consume_rows16(A, bu, bu + 2 * kRowHalf, it.n,
                   it.type == IT_SUM ? bias + (it.a - C.k0) : nullptr, P.scale_log2);
  } else {
    int off_key = -1, off_uk = 0, off_uv = 0, off_val = -1, n = 0;
    if (it.type == IT_REC) {
      const RecordLayout L = record_layout(it.n, it.rk, it.rv);
      off_key = 0;
      off_uk = int(L.uk);
      off_uv = int(L.uv);
      off_val = int(L.vpart);
      n = it.n;
    } else if (it.type == IT_KEY) {
      off_key = 0;
    } else if (it.type == IT_UT) {
      off_uv = it.uv;
      n = it.n;
    } else {
      off_val = 0;
    }
    if (off_key >= 0) exp_key<KS>(A, X, base + off_key, it.rk, P.scale_log2);
    if (n > 0) exp_tokens<KS>(A, X, base + off_uk, base + off_uv, n, it.rk, it.rv);
    if (off_val >= 0) exp_value<KS>(A, X, base + off_val, it.rv);
  }
  __syncwarp();
  Q.tail = it.end;
  ++Q.nd;
}

// Routing page p of this CTA (fused mode), landed as the warp's next item:
// expansion decisions for its spans, their summary biases and record entries.
__device__ __forceinline__ void route_page(uint8_t* smem, SmemMisc* ms, const Ctx& C,
                                           const DecodeParams& P, WarpQ& Q, int p, int body,
                                           int rank, long long off) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const float* ys = reinterpret_cast<const float*>(smem + kOffY);
  float* bias = reinterpret_cast<float*>(smem + kOffBias);
  RecEntry* ents = reinterpret_cast<RecEntry*>(smem + kOffEntries);
  bool hit = false;
  int end = 0;
  if (Q.ok) {
    if (wait_item(ms, Q)) {
      const Item it = ms->desc[w][Q.nd % kMaxItems];
      end = it.end;
      hit = route32(smem + it.boff, ys, ms->theta, P.G);
    } else {
      if (lane == 0) set_device_error(P.status, DEV_WAIT_TIMEOUT, 5);
      Q.ok = 0;
    }
  }
  const int k = C.k0 + kRouteSpans * p + lane;
  const bool valid = k < C.k1;
  const bool ex = valid && body > 0 && hit;
  if (valid) bias[k - C.k0] = (body > 0 && !ex) ? log2f(float(body)) : kNegInf;
  const uint32_t bal = __ballot_sync(kFull, ex);
  int base = 0;
  if (lane == 0) {
    ms->pmask[p] = bal;
    base = bal ? atomicAdd(&ms->n_rec, __popc(bal)) : 0;
  }
  base = __shfl_sync(kFull, base, 0);
  if (ex) {
    RecEntry en;
    en.off_lo = int(uint32_t(off));
    en.off_hi = int(off >> 32);
    en.body = body;
    en.rank = rank;
    ents[base + __popc(bal & ((1u << lane) - 1u))] = en;
  }
  __syncwarp();
  if (Q.ok) {
    Q.tail = end;
    ++Q.nd;
  }
}

// Issue routing page p (fused mode) as the warp's next item; the arena is
// empty or holds only earlier routing pages, so it always fits.
__device__ __forceinline__ void issue_route_page(uint8_t* smem, SmemMisc* ms, const Ctx& C,
                                                 const DecodeParams& P, WarpQ& Q, int p) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int start = arena_place(Q, kRoutePageBytes);
  Item it{};
  it.type = IT_ROUTE;
  it.a = C.k0 + kRouteSpans * p;
  it.boff = kOffArena + w * kArenaBytes + (start % kArenaGran) * kGran;
  it.end = start + kRoutePageBytes / kGran;
  const int slot = Q.ni % kMaxItems;
  if (lane == 0) {
    arm_item(ms, w, slot, it, kRoutePageBytes);
    tma_g2s_4d_hint(smem + it.boff, &P.tm_sroute, 0, it.a, 0, C.g, &ms->bar[w][slot],
                    policy_evict_first());
  }
  Q.head = it.end;
  ++Q.ni;
}

template <int KS>
__device__ __forceinline__ void run_decode(uint8_t* smem, SmemMisc* ms, const DecodeParams& P) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  Ctx C;
  C.j = blockIdx.x;
  C.c = blockIdx.y;
  C.b = blockIdx.z;
  C.g = C.b * P.Hkv + C.c;
  C.gs = size_t(C.g) * P.max_spans;
  C.bs = size_t(C.b) * P.max_spans;
  const int n_sp = P.n_spans[C.b];
  const int n_full = P.n_sink + n_sp + P.n_recent;
  fixed_range(C.j, P.cg, n_full, n_sp, C.f0, C.f1, C.k0, C.k1);
  C.nfp = (C.f1 - C.f0 + kRows - 1) / kRows;
  C.n_fixed = C.nfp + (C.k1 - C.k0 + kRows - 1) / kRows;
  C.n_rp = P.fused ? (C.k1 - C.k0 + kRouteSpans - 1) / kRouteSpans : 0;
  const int G = P.G;

  WarpQ Q{};
  Q.ok = 1;
  if (lane == 0) {
    prefetch_tmap(&P.tm_kfull);
    prefetch_tmap(&P.tm_vfull);
    prefetch_tmap(&P.tm_ksum);
    prefetch_tmap(&P.tm_vsum);
    if (P.fused) prefetch_tmap(&P.tm_sroute);
  }

  // ---- prologue: routing pages and the first fixed pages (no q needed) ----
  // routing pages p = w, w + 8 of this CTA, with their spans' metadata
  int rbody[2] = {0, 0}, rrank[2] = {0, 0};
  long long roff[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int p = w + kWarps * i;
    if (p < C.n_rp) {
      issue_route_page(smem, ms, C, P, Q, p);
      const int k = C.k0 + kRouteSpans * p + lane;
      if (k < C.k1) {
        rbody[i] = __ldg(P.body_len + C.bs + k);
        rrank[i] = __ldg(P.rec_rank + C.gs + k);
        roff[i] = __ldg(reinterpret_cast<const long long*>(P.rec_off) + C.gs + k);
      }
    }
  }
  // y = W_r q, rows 8w .. 8w + 7 of this warp: lane (r = lane / 4, quarter
  // d = lane % 4) takes 32 of the 128 head dims; W_r is read before the
  // dependency wait (the caller allows it), q after
  float4 wr[8];
  if (P.fused) {
    const float4* wrow = reinterpret_cast<const float4*>(
        P.W_r + (size_t(C.c) * kRouteDim + 8 * w + (lane >> 2)) * kHeadDim + 32 * (lane & 3));
#pragma unroll
    for (int i = 0; i < 8; ++i) wr[i] = __ldg(wrow + i);
  }
  issue_more(smem, ms, P, C, Q, false);

  // ---- the query (and in list mode the lists) come from earlier work ------
  pdl_wait();
  float* qf = reinterpret_cast<float*>(smem + kOffQf);
  {
    // q as f32 [8][128] (rows past the group zero) for the routing projection
    const int h = tid >> 5, d = 4 * (tid & 31);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h < G) {
      const __nv_bfloat16* qr = P.q + (size_t(C.b) * P.Hq + size_t(C.c) * G + h) * kHeadDim + d;
      const uint2 u = *reinterpret_cast<const uint2*>(qr);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      v = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    *reinterpret_cast<float4*>(qf + h * kHeadDim + d) = v;
  }
  if (w == 0) {
    // query A fragments (rows 0..7 = heads, zero past G), grouped by 32 dims
    const int r0 = lane >> 2;
    const __nv_bfloat16* qg = P.q + (size_t(C.b) * P.Hq + size_t(C.c) * G) * kHeadDim;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = 32 * i + 2 * (lane & 3);
      const __nv_bfloat16* qr = qg + r0 * kHeadDim + k;
      uint4 v;
      v.x = r0 < G ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
      v.y = r0 < G ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
      v.z = r0 < G ? *reinterpret_cast<const uint32_t*>(qr + 16) : 0u;
      v.w = r0 < G ? *reinterpret_cast<const uint32_t*>(qr + 24) : 0u;
      sts128(smem_u32(smem + kOffQfrag) + (i * 32 + lane) * 16, v);
    }
  }
  if (P.fused && tid < 8) ms->theta[tid] = tid < G ? P.theta[C.c * G + tid] : 0.f;
  __syncthreads();

  if (P.fused) {
    float* ys = reinterpret_cast<float*>(smem + kOffY);
    float acc[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[h] = 0.f;
    const int dq = lane & 3;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float4 qv = *reinterpret_cast<const float4*>(qf + h * kHeadDim + 32 * dq + 4 * i);
        acc[h] = fmaf(wr[i].w, qv.w, fmaf(wr[i].z, qv.z, fmaf(wr[i].y, qv.y,
                      fmaf(wr[i].x, qv.x, acc[h]))));
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      acc[h] += __shfl_xor_sync(kFull, acc[h], 1);
      acc[h] += __shfl_xor_sync(kFull, acc[h], 2);
    }
    if (dq == 0) {
#pragma unroll
      for (int h = 0; h < 8; ++h) ys[h * kRouteDim + 8 * w + (lane >> 2)] = acc[h];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int p = w + kWarps * i;
      if (p < C.n_rp) route_page(smem, ms, C, P, Q, p, rbody[i], rrank[i], roff[i]);
    }
  } else {
    // list mode: this CTA's expanded spans from the caller's ascending list
    // (every CTA checks the whole list; the first error wins)
    RecEntry* ents = reinterpret_cast<RecEntry*>(smem + kOffEntries);
    int n = P.list_n[C.g];
    if (n < 0 || n > n_sp) {
      if (tid == 0) set_device_error(P.status, DEV_BAD_LIST, C.g);
      n = 0;
    }
    for (int e = tid; e < n; e += kThreads) {
      const int k = P.list[C.gs + e];
      const int prev = e > 0 ? P.list[C.gs + e - 1] : -1;
      bool ok = k > prev && k < n_sp;
      int body = 0, rank = 0;
      if (ok) {
        body = P.body_len[C.bs + k];
        rank = P.rec_rank[C.gs + k];
        ok = body > 0;
      }
      if (!ok) {
        set_device_error(P.status, DEV_BAD_LIST, e);
      } else if (k >= C.k0 && k < C.k1) {
        // a span enters once even if a malformed list names it twice, so the
        // entries never outgrow the CTA's share
        const uint32_t bit = 1u << ((k - C.k0) & 31);
        if (atomicOr(&ms->pmask[(k - C.k0) >> 5], bit) & bit) {
          set_device_error(P.status, DEV_BAD_LIST, e);
        } else {
          const long long off = P.staged_off != nullptr ? P.staged_off[C.gs + e]
                                                        : P.rec_off[C.gs + k];
          RecEntry en;
          en.off_lo = int(uint32_t(off));
          en.off_hi = int(off >> 32);
          en.body = body;
          en.rank = rank;
          ents[atomicAdd(&ms->n_rec, 1)] = en;
        }
      }
    }
    __syncthreads();
    float* bias = reinterpret_cast<float*>(smem + kOffBias);
    for (int i = tid; i < C.k1 - C.k0; i += kThreads) {
      const int body = P.body_len[C.bs + C.k0 + i];
      const bool ex = (ms->pmask[i >> 5] >> (i & 31)) & 1u;
      bias[i] = (body > 0 && !ex) ? log2f(float(body)) : kNegInf;
    }
  }
  __syncthreads();  // routing barrier: biases and the record list are final

  if (P.fused && w == 0 && P.expanded_out != nullptr) {
    // this CTA's expanded spans, ascending, for the group's output list
    int cnt = 0;
    for (int p0 = 0; p0 < C.n_rp; p0 += 32) {
      const int p = p0 + lane;
      const uint32_t m = p < C.n_rp ? ms->pmask[p] : 0u;
      const int c = __popc(m);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
      }
      int pos = cnt + incl - c;
      for (uint32_t mm = m; mm; mm &= mm - 1)
        P.cta_list[C.gs + C.k0 + pos++] = C.k0 + kRouteSpans * p + __ffs(mm) - 1;
      cnt += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) P.cta_n[size_t(C.g) * P.cg + C.j] = cnt;
  }

  // ---- main loop: issue, wait, consume --------------------------------------
  WarpAcc A;
  A.qfrag = smem_u32(smem + kOffQfrag);
#pragma unroll
  for (int t = 0; t < 16; ++t) A.o[t][0] = A.o[t][1] = 0.f;
  A.m_row = kNegInf;
  A.l_part = 0.f;
  ExpAcc<KS> X;
  X.had = false;
  for (;;) {
    issue_more(smem, ms, P, C, Q, true);
    if (Q.nd == Q.ni || !Q.ok) break;
    if (!wait_item(ms, Q)) {
      if (lane == 0) set_device_error(P.status, DEV_WAIT_TIMEOUT, 4);
      Q.ok = 0;
      break;
    }
    consume_item<KS>(smem, ms, C, P, Q, A, X);
  }
  // after a timeout: every issued copy lands before the arena is reused
  for (; Q.nd < Q.ni; ++Q.nd) {
    if (!mbar_wait(&ms->bar[w][Q.nd % kMaxItems], uint32_t((Q.nd / kMaxItems) & 1),
                   kWaitLimit)) {
      if (lane == 0) set_device_error(P.status, DEV_WAIT_TIMEOUT, 3);
      break;
    }
  }

  // ---- merge the eight warps' states into this CTA's partial --------------
  // (each warp writes into its own arena, which is idle now)
  {
    float* wst = reinterpret_cast<float*>(smem + kOffArena + w * kArenaBytes);  // m[8] l[8] o[8][128]
    const int r0 = lane >> 2;
    float l_row = A.l_part + __shfl_xor_sync(kFull, A.l_part, 1);
    l_row += __shfl_xor_sync(kFull, l_row, 2);
    if ((lane & 3) == 0) {
      wst[r0] = r0 < G ? A.m_row : kNegInf;
      wst[8 + r0] = r0 < G ? l_row : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      wst[16 + r0 * kHeadDim + 8 * t + 2 * (lane & 3)] = A.o[t][0];
      wst[16 + r0 * kHeadDim + 8 * t + 2 * (lane & 3) + 1] = A.o[t][1];
    }
  }
  __syncthreads();
  Partial* mine = P.partials + size_t(C.g) * P.cg + C.j;
  {
    const int d = tid & (kHeadDim - 1);
    for (int h = tid >> 7; h < G; h += 2) {
      float M = kNegInf;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww)
        M = fmaxf(M, reinterpret_cast<const float*>(smem + ww * kArenaBytes)[h]);
      float L = 0.f, O = 0.f;
      if (M != kNegInf) {
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) {
          const float* ws_ = reinterpret_cast<const float*>(smem + ww * kArenaBytes);
          const float sc = exp2f(ws_[h] - M);
          L = fmaf(ws_[8 + h], sc, L);
          O = fmaf(ws_[16 + h * kHeadDim + d], sc, O);
        }
      }
      mine->o[h][d] = O;
      if (d == 0) {
        mine->m[h] = M;
        mine->l[h] = L;
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int old = atomicAdd(&P.groups[C.g].done, 1);
    ms->is_last = (old == P.cg - 1);
  }
  __syncthreads();
  if (!ms->is_last) return;

  // ---- last CTA of this group: merge the partials, write the output --------
  __threadfence();
  const int cg = P.cg;
  const Partial* parts = P.partials + size_t(C.g) * cg;
  float* sm_m = reinterpret_cast<float*>(smem);                 // [cg][8] m, then scales
  float* sm_l = sm_m + kMaxCg * 8;                              // [cg][8] l
  float* sm_ML = sm_l + kMaxCg * 8;                             // M[8], L[8]
  for (int i = tid; i < cg * 8; i += kThreads) {
    const int jj = i >> 3, h = i & 7;
    sm_m[i] = h < G ? __ldcg(&parts[jj].m[h]) : kNegInf;
    sm_l[i] = h < G ? __ldcg(&parts[jj].l[h]) : 0.f;
  }
  __syncthreads();
  if (tid < 8) {
    float M = kNegInf;
    for (int jj = 0; jj < cg; ++jj) M = fmaxf(M, sm_m[jj * 8 + tid]);
    float L = 0.f;
    if (M != kNegInf)
      for (int jj = 0; jj < cg; ++jj) L = fmaf(sm_l[jj * 8 + tid], exp2f(sm_m[jj * 8 + tid] - M), L);
    sm_ML[tid] = M;
    sm_ML[8 + tid] = L;
  }
  __syncthreads();
  for (int i = tid; i < cg * 8; i += kThreads) {
    const float M = sm_ML[i & 7];
    sm_m[i] = (M == kNegInf) ? 0.f : exp2f(sm_m[i] - M);
  }
  __syncthreads();
  {
    const int d = tid & (kHeadDim - 1);
    for (int h = tid >> 7; h < G; h += 2) {
      float O = 0.f;
#pragma unroll 4
      for (int jj = 0; jj < cg; ++jj) O = fmaf(__ldcg(&parts[jj].o[h][d]), sm_m[jj * 8 + h], O);
      const float L = sm_ML[8 + h];
      const size_t row = size_t(C.b) * P.Hq + size_t(C.c) * G + h;
      P.out[row * kHeadDim + d] = L > 0.f ? O / L : 0.f;
      if (d == 0 && P.lse != nullptr)
        P.lse[row] = L > 0.f ? (sm_ML[h] + log2f(L)) * kLn2 : kNegInf;
    }
  }
  if (P.fused && P.expanded_out != nullptr) {
    // the CTAs' ascending lists, one after the other
    int* pre = reinterpret_cast<int*>(sm_ML + 16);  // [cg + 1]
    if (tid == 0) {
      int acc = 0;
      for (int jj = 0; jj < cg; ++jj) {
        pre[jj] = acc;
        acc += __ldcg(P.cta_n + size_t(C.g) * cg + jj);
      }
      pre[cg] = acc;
    }
    __syncthreads();
    for (int jj = w; jj < cg; jj += kWarps) {
      int a0, a1, sk0, sk1;
      fixed_range(jj, cg, n_full, n_sp, a0, a1, sk0, sk1);
      const int cnt = pre[jj + 1] - pre[jj];
      for (int i = lane; i < cnt; i += 32)
        P.expanded_out[C.gs + pre[jj] + i] = __ldcg(P.cta_list + C.gs + sk0 + i);
    }
    if (tid == 0 && P.n_expanded_out != nullptr) P.n_expanded_out[C.g] = pre[cg];
  }
  __syncthreads();
  if (tid == 0) P.groups[C.g].done = 0;
}

// grid: (cg, Hkv, B); block: 8 warps, each its own producer and consumer
template <int KS>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  SmemMisc* ms = reinterpret_cast<SmemMisc*>(smem + kOffMisc);
  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w)
      for (int s = 0; s < kMaxItems; ++s) mbar_init(&ms->bar[w][s], 1);
    ms->n_rec = 0;
    ms->rec_next = 0;
    ms->fixed_next = 0;
    ms->is_last = 0;
    for (int p = 0; p < kMaxRoutePages; ++p) ms->pmask[p] = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  run_decode<KS>(smem, ms, P);
}

}  // namespace sekv
