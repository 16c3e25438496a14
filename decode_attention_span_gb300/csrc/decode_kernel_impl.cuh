// The decode kernel's body, a template on KS (rank k-steps of 16: ranks up
// to 16 KS).  Each KS is instantiated in a translation unit of its own.
//
// Per warp: an arena of kArenaGran granules used as a ring (items are placed
// contiguously, wrapping to the arena start when one does not fit at the
// end), up to kMaxItems items in flight (before routing: its routing pages
// and the first own pages, kPrologueItems in all), each with its own
// mbarrier.  The
// warp issues and consumes its items itself, in order, so no handover
// between warps is needed; the only CTA-wide synchronisation is the routing
// barrier (every span of the CTA routed, the record list final) and the
// merge at the end.  Lane 0 alone runs the issue logic, on the warp's state
// in shared memory, so the consuming lanes keep their registers for the
// softmax state and the kernel needs no stack.
#pragma once

#include "decode_consumer.cuh"

namespace sekv {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Place an item of `bytes` in a warp's arena: returns the granule counter of
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

// Arm item `it` (lane 0): descriptor, then the barrier with its bytes; the
// caller issues its copies next.  The descriptor is published by the
// barrier's phase completion, which the consuming lanes acquire when they
// wait on it.
__device__ __forceinline__ void arm_item(SmemMisc* ms, int w, int slot, const Item& it,
                                         uint32_t bytes) {
  ms->desc[w][slot] = it;
  // the warp's earlier reads of this arena space (generic proxy) come
  // before the copies that overwrite it (async proxy)
  fence_proxy_async_smem();
  mbar_arrive_expect_tx(&ms->bar[w][slot], bytes);
}

// The entry of an expanded span: its record's parts (1 if it lands whole)
// and U rows per tile; a rank above the instance's limit is flagged here and
// the entry gets 0 parts (skipped).
__device__ __forceinline__ RecEntry rec_entry(const DecodeParams& P, long long off, int body,
                                              unsigned cols, int rank, int& parts) {
  const int rK = rank & 0xffff, rV = (rank >> 16) & 0xffff;
  int rows16 = 0;
  parts = 0;
  if (rK > P.rank_lim || rV > P.rank_lim) {
    set_device_error(P.status, DEV_BAD_RANK, rK > rV ? rK : rV);
  } else {
    parts = record_parts(body, rK, rV);  // no division for a record that lands whole
    if (parts > 1) rows16 = split_rows(rK, rV) >> 4;
  }
  RecEntry en;
  en.off_lo = int(uint32_t(off));
  en.off_hi = int(off >> 32);
  en.body = body | int(cols << 16) | (parts << 24);
  en.rank = (rK & 0xff) | (rows16 << 8) | ((rV & 0xff) << 16);
  return en;
}

// Issue the warp's next items while it has room (lane 0, on a register copy
// of the warp's state): first any claim still pending, then new claims.
// Before routing is done only the CTA's own pages, at most kPrologueItems
// items; after it, records, then own pages, then the group's pool.  Pool
// claims are made one ahead: `claim` holds the pending atomic's result, so
// its round trip overlaps the warp's work (-1: none made yet).
__device__ __forceinline__ void issue_more(uint8_t* smem, SmemMisc* ms, const DecodeParams& P,
                                           bool routed, int& claim) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) {
    WarpQ Q = ms->wq[w];
    const Ctx C = ms->ctx;
    const int n_front = ms->n_front, n_rec = n_front + ms->n_back;
    const int cap = routed ? kMaxItems : kPrologueItems;
    const RecEntry* ents = reinterpret_cast<const RecEntry*>(smem + kOffEntries);
    const uint64_t pol = policy_evict_first();
    while (Q.ok && Q.ni - Q.nd < cap) {
      if (Q.pk == 0 && routed && !Q.rec_out) {
        const int e = atomicAdd(&ms->rec_next, 1);
        if (e < n_rec) {
          const int ei = rec_slot(e, n_front);
          const int parts = (ents[ei].body >> 24) & 0xff;
          if (parts == 0) continue;  // skipped (flagged when the entry was made)
          Q.pk = 2;
          Q.pidx = ei;
          Q.ppart = 0;
          Q.pnp = parts;
        } else {
          Q.rec_out = 1;
        }
      }
      if (Q.pk == 0 && !Q.fixed_out) {
        const int f = atomicAdd(&ms->fixed_next, 1);
        if (f < C.n_fixed) {
          Q.pk = 1;
          Q.pidx = f;
        } else {
          Q.fixed_out = 1;
        }
      }
      if (Q.pk == 0 && routed && !Q.pool_out) {
        if (claim < 0) claim = atomicAdd(&P.groups[C.g].full_next, kPoolClaim);
        const int first = C.pool0 + claim;
        if (first < C.n_fp) {
          Q.pk = 3;
          Q.pidx = first;
          Q.ppart = 0;
          Q.pnp = (C.n_fp - first) < kPoolClaim ? (C.n_fp - first) : kPoolClaim;
          claim = atomicAdd(&P.groups[C.g].full_next, kPoolClaim);  // the next one, ahead
        } else {
          Q.pool_out = 1;
        }
      }
      if (Q.pk == 0) break;

      Item it{};
      uint32_t bytes = 0;
      int64_t s0 = 0, s1 = 0;
      uint32_t n0 = 0, n1 = 0;
      int64_t roff = 0;
      if (Q.pk != 2) {
        const bool full = Q.pk == 3 || Q.pidx < C.n_own;
        it.type = full ? IT_FULL : IT_SUM;
        it.a = Q.pk == 3 ? kFullRows * (Q.pidx + Q.ppart)
                         : (full ? kFullRows * (C.own0 + Q.pidx) : C.k0 + kRows * (Q.pidx - C.n_own));
        const int e = full ? C.n_full : C.k1, rows = full ? kFullRows : kRows;
        it.n = (e - it.a) < rows ? (e - it.a) : rows;
        bytes = full ? kFullPageBytes : kRowPageBytes;
      } else {
        const RecEntry en = ents[Q.pidx];
        const int b = en.body & 0xffff, rK = en.rank & 0xff, rV = (en.rank >> 16) & 0xff;
        const RecordLayout L = record_layout(b, rK, rV);
        roff = (int64_t(uint32_t(en.off_lo)) | (int64_t(en.off_hi) << 32));
        it.rk = rK;
        it.rv = rV;
        it.a = (en.body >> 16) & 0xff;  // the query columns that expand the span
        if (Q.pnp == 1) {
          it.type = IT_REC;
          it.n = b;
          n0 = uint32_t(L.total);
        } else if (Q.ppart == 0) {
          it.type = IT_KEY;
          n0 = uint32_t(L.uk);
        } else if (Q.ppart < Q.pnp - 1) {
          const int rows = ((en.rank >> 8) & 0xff) << 4;
          const int i0 = (Q.ppart - 1) * rows;
          it.type = IT_UT;
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
      const int slot = Q.ni % kSlots;
      const int gsz = int((bytes + kGran - 1) / kGran);
      it.boff = kOffArena + w * kArenaBytes + (start % kArenaGran) * kGran;
      it.end = start + gsz;
      arm_item(ms, w, slot, it, bytes);
      uint8_t* dst = smem + it.boff;
      uint64_t* bar = &ms->bar[w][slot];
      if (Q.pk != 2) {
        const bool full = it.type == IT_FULL;
        tma_g2s_4d_hint(dst, full ? &P.tm_kfull : &P.tm_ksum, 0, it.a, 0, C.g, bar, pol);
        tma_g2s_4d_hint(dst + (full ? 2 * kFullHalf : 2 * kRowHalf), full ? &P.tm_vfull : &P.tm_vsum,
                        0, it.a, 0, C.g, bar, pol);
      } else {
        const uint8_t* rec = P.store + roff;
        if (n0) bulk_g2s_hint(dst, rec + s0, n0, bar, pol);
        if (n1) bulk_g2s_hint(dst + n0, rec + s1, n1, bar, pol);
      }
      Q.head = it.end;
      ++Q.ni;
      if (Q.pk == 1 || ++Q.ppart == Q.pnp) Q.pk = 0;
    }
    ms->wq[w] = Q;
  }
  __syncwarp();
}

// Consume the warp's item nd (landed); returns its end in the arena.
template <int KS, bool MQ>
__device__ __forceinline__ int consume_item(const uint8_t* smem, SmemMisc* ms,
                                            const DecodeParams& P, int nd, WarpAcc& A,
                                            ExpAcc<KS>& X) {
  const int w = threadIdx.x >> 5;
  const Item it = ms->desc[w][nd % kSlots];
  const uint8_t* base = smem + it.boff;
  const uint32_t bu = smem_u32(base);
  const float* bias = reinterpret_cast<const float*>(smem + kOffBias);
  if (it.type == IT_FULL) {
    consume_rows32(A, bu, bu + 2 * kFullHalf, it.n, P.scale_log2, kFullHalf);
  } else if (it.type == IT_SUM) {
    consume_rows16<MQ>(A, bu, bu + 2 * kRowHalf, it.n, bias + (it.a - ms->ctx.k0),
                       P.scale_log2, kRowHalf, smem + kOffCmask + (it.a - ms->ctx.k0));
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
    if (n > 0) exp_tokens<KS, MQ>(A, X, base + off_uk, base + off_uv, n, it.rk, it.rv, unsigned(it.a));
    if (off_val >= 0) exp_value<KS>(A, X, base + off_val, it.rv);
  }
  return it.end;
}

// The warp's item nd is consumed and its arena space free (lane 0 records it).
__device__ __forceinline__ void retire_item(SmemMisc* ms, int nd, int end) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    WarpQ& Q = ms->wq[threadIdx.x >> 5];
    Q.tail = end;
    Q.nd = nd + 1;
  }
}

// Issue routing page p (fused mode, lane 0) as the warp's next item; the
// arena is empty or holds only earlier routing pages, so it always fits.
__device__ __forceinline__ void issue_route_page(uint8_t* smem, SmemMisc* ms,
                                                 const DecodeParams& P, int p) {
  const int w = threadIdx.x >> 5;
  WarpQ& Q = ms->wq[w];
  const Ctx& C = ms->ctx;
  const int start = arena_place(Q, kRoutePageBytes);
  Item it{};
  it.type = IT_ROUTE;
  it.a = C.k0 + kRouteSpans * p;
  it.boff = kOffArena + w * kArenaBytes + (start % kArenaGran) * kGran;
  it.end = start + kRoutePageBytes / kGran;
  const int slot = Q.ni % kSlots;
  arm_item(ms, w, slot, it, kRoutePageBytes);
  tma_g2s_4d_hint(smem + it.boff, &P.tm_sroute, 0, it.a, 0, C.g, &ms->bar[w][slot],
                  policy_evict_first());
  Q.head = it.end;
  ++Q.ni;
}

// Routing page p of this CTA (fused mode), landed as the warp's next item:
// expansion decisions for its spans, their summary biases and record entries.
template <bool MQ>
__device__ __forceinline__ void route_page(uint8_t* smem, SmemMisc* ms, const DecodeParams& P,
                                           int p, int body, int rank, long long off) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const float* ys = reinterpret_cast<const float*>(smem + kOffY);
  float* bias = reinterpret_cast<float*>(smem + kOffBias);
  RecEntry* ents = reinterpret_cast<RecEntry*>(smem + kOffEntries);
  const int nd = ms->wq[w].nd;
  const int k0 = ms->ctx.k0, k1 = ms->ctx.k1;
  unsigned cols = 0u;  // the query columns whose gate logit passes their threshold
  bool landed = false;
  int end = 0;
  if (ms->wq[w].ok) {
    landed = mbar_wait_parked(&ms->bar[w][nd % kSlots], uint32_t((nd / kSlots) & 1), P.wait_ns);
    if (landed) {
      const Item it = ms->desc[w][nd % kSlots];
      end = it.end;
      cols = route32(smem + it.boff, ys, ms->theta, P.G);
    } else if (lane == 0) {
      set_device_error(P.status, DEV_WAIT_TIMEOUT, 5);
    }
  }
  // a query token expands the span if any of its heads does (the union over
  // the group); its columns then see the reconstructed tokens and not the
  // summary
  const unsigned all = (1u << P.G) - 1u;
  unsigned cm = cols != 0u ? all : 0u;  // one token: every column or none
  if (MQ) {
    const unsigned tok = (1u << P.hpg) - 1u;
    cm = 0u;
    for (int i = 0; i < P.nq; ++i)
      if ((cols >> (i * P.hpg)) & tok) cm |= tok << (i * P.hpg);
  }
  const int k = k0 + kRouteSpans * p + lane;
  const bool valid = k < k1;
  if (!(valid && body > 0)) cm = 0u;
  const bool ex = cm != 0u;
  if (valid) bias[k - k0] = (body > 0 && cm != all) ? log2f(float(body)) : kNegInf;
  if (MQ && valid) smem[kOffCmask + (k - k0)] = uint8_t(cm);
  // records that arrive in parts go to the front of the queue, the others to
  // its back (longest first: a split record is one warp's serial chain)
  int parts = 0;
  RecEntry en{};
  if (ex) en = rec_entry(P, off, body, cm, rank, parts);
  const bool big = parts > 1;
  const uint32_t bal = __ballot_sync(kFull, ex);
  const uint32_t bbig = __ballot_sync(kFull, big), bsmall = bal & ~bbig;
  int bf = 0, bb = 0;
  if (lane == 0) {
    ms->pmask[p] = bal;
    if (bbig) bf = atomicAdd(&ms->n_front, __popc(bbig));
    if (bsmall) bb = atomicAdd(&ms->n_back, __popc(bsmall));
  }
  bf = __shfl_sync(kFull, bf, 0);
  bb = __shfl_sync(kFull, bb, 0);
  if (ex) {
    const uint32_t below = (1u << lane) - 1u;
    ents[big ? bf + __popc(bbig & below) : kSpanCap - 1 - (bb + __popc(bsmall & below))] = en;
  }
  if (landed) {
    retire_item(ms, nd, end);
  } else {
    __syncwarp();
    if (lane == 0) ms->wq[w].ok = 0;
  }
  __syncwarp();
}

template <int KS, bool MQ>
__device__ __forceinline__ void run_decode(uint8_t* smem, SmemMisc* ms, const DecodeParams& P,
                                           const float4 (&wr)[8]) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const Ctx& C = ms->ctx;
  const int G = P.G;

  // ---- prologue: routing pages and the first own pages (no q needed; the
  // routing weights `wr` were requested at kernel entry) ---------------------
  const int wr_r = lane >> 2, wr_dq = lane & 3;
  if (lane == 0) {
    for (int p = w; p < C.n_rp; p += kWarps) issue_route_page(smem, ms, P, p);
  }
  int claim = -1;  // lane 0: the next pool claim, made ahead
  issue_more(smem, ms, P, false, claim);
  // the metadata of this warp's routing pages (p = w, w + 8)
  int rbody[2] = {0, 0}, rrank[2] = {0, 0};
  long long roff[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int k = C.k0 + kRouteSpans * (w + kWarps * i) + lane;
    if (w + kWarps * i < C.n_rp && k < C.k1) {
      rbody[i] = __ldg(P.body_len + C.bs + k);
      rrank[i] = __ldg(P.rec_rank + C.gs + k);
      roff[i] = __ldg(reinterpret_cast<const long long*>(P.rec_off) + C.gs + k);
    }
  }

  // ---- the query (and in list mode the lists) come from earlier work ------
  pdl_wait();
  float* qf = reinterpret_cast<float*>(smem + kOffQf);
  {
    // one round trip: thread t loads q[h][d .. d + 3] (h = t / 32, d = 4 (t % 32);
    // rows past the group read as zero) and, for t < 8, theta.  It stores
    // them as f32 for the routing projection and as the bf16 pairs of the
    // query's mma A fragments (rows 0..7 = heads, grouped by 32 dims: pair
    // (h, 32 i + 8 k + 2 j) is component k of lane 4 h + j's fragment i).
    // (column h: query token h / hpg, head h % hpg; q is [B][nq][Hq][128])
    const int h = tid >> 5, d = 4 * (tid & 31);
    uint2 u = make_uint2(0u, 0u);
    const int hq = MQ ? (C.b * P.nq_all + h / P.hpg) * P.Hq + C.c * P.hpg + h % P.hpg
                      : C.b * P.Hq + C.c * G + h;
    if (h < G) u = *reinterpret_cast<const uint2*>(P.q + size_t(hq) * kHeadDim + d);
    const float th = (P.fused && tid < G) ? P.theta[C.c * P.hpg + (MQ ? tid % P.hpg : tid)] : 0.f;
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    *reinterpret_cast<float4*>(qf + h * kHeadDim + d) = make_float4(lo.x, lo.y, hi.x, hi.y);
    uint32_t* qfr = reinterpret_cast<uint32_t*>(smem + kOffQfrag);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int dd = d + 2 * e, i = dd >> 5, k = (dd & 31) >> 3, j = (dd & 7) >> 1;
      qfr[(i * 32 + 4 * h + j) * 4 + k] = e ? u.y : u.x;
    }
    if (tid < 8) ms->theta[tid] = th;
  }
  __syncthreads();

  if (P.fused) {
    // y = W_r q, rows 8w .. 8w + 7 of this warp, from the registers: at step
    // i lane (r, dq) multiplies chunk dq + 4 i of its row with the same chunk
    // of each head's query, which the 8 lanes of equal dq read together (one
    // broadcast shared-memory wavefront per read)
    float* ys = reinterpret_cast<float*>(smem + kOffY);
    float acc[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[h] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = wr_dq + 4 * i;
      const float4 wv = wr[i];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h < G) {
          const float4 qv = *reinterpret_cast<const float4*>(qf + h * kHeadDim + 4 * c);
          acc[h] = fmaf(wv.w, qv.w, fmaf(wv.z, qv.z, fmaf(wv.y, qv.y, fmaf(wv.x, qv.x, acc[h]))));
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      acc[h] += __shfl_xor_sync(kFull, acc[h], 1);
      acc[h] += __shfl_xor_sync(kFull, acc[h], 2);
    }
    if (wr_dq == 0) {
#pragma unroll
      for (int h = 0; h < 8; ++h) ys[h * kRouteDim + 8 * w + wr_r] = acc[h];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int p = w + kWarps * i;
      if (p < C.n_rp) route_page<MQ>(smem, ms, P, p, rbody[i], rrank[i], roff[i]);
    }
  } else {
    // list mode: this CTA's expanded spans from the caller's ascending list
    // (every CTA checks the whole list; the first error wins)
    RecEntry* ents = reinterpret_cast<RecEntry*>(smem + kOffEntries);
    int n = P.list_n[C.g];
    if (n < 0 || n > C.n_sp) {
      if (tid == 0) set_device_error(P.status, DEV_BAD_LIST, C.g);
      n = 0;
    }
    for (int e = tid; e < n; e += kThreads) {
      const int k = P.list[C.gs + e];
      const int prev = e > 0 ? P.list[C.gs + e - 1] : -1;
      bool ok = k > prev && k < C.n_sp;
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
          int parts;
          const RecEntry en = rec_entry(P, off, body, (1u << P.G) - 1u, rank, parts);  // every column
          if (parts > 1)
            ents[atomicAdd(&ms->n_front, 1)] = en;
          else
            ents[kSpanCap - 1 - atomicAdd(&ms->n_back, 1)] = en;
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
  for (int t = 0; t < 8; ++t) A.o[t][0] = A.o[t][1] = A.o[t][2] = A.o[t][3] = 0.f;
  A.m[0] = A.m[1] = kNegInf;
  A.l[0] = A.l[1] = 0.f;
  ExpAcc<KS> X;
  X.had = false;
  for (;;) {
    issue_more(smem, ms, P, true, claim);
    const int nd = ms->wq[w].nd;
    if (nd == ms->wq[w].ni || !ms->wq[w].ok) break;
    if (!mbar_wait_parked(&ms->bar[w][nd % kSlots], uint32_t((nd / kSlots) & 1), P.wait_ns)) {
      __syncwarp();
      if (lane == 0) {
        set_device_error(P.status, DEV_WAIT_TIMEOUT, 4);
        ms->wq[w].ok = 0;
      }
      __syncwarp();
      break;
    }
    const int end = consume_item<KS, MQ>(smem, ms, P, nd, A, X);
    retire_item(ms, nd, end);
  }
  // after a timeout: every issued copy lands before the arena is reused
  {
    const int ni = ms->wq[w].ni;
    for (int nd = ms->wq[w].nd; nd < ni; ++nd) {
      if (!mbar_wait(&ms->bar[w][nd % kSlots], uint32_t((nd / kSlots) & 1),
                     kWaitLimit)) {
        if (lane == 0) set_device_error(P.status, DEV_WAIT_TIMEOUT, 3);
        break;
      }
    }
  }

  // ---- merge the eight warps' states into this CTA's partial --------------
  // (each warp writes into its own arena, which is idle now)
  {
    float* wst = reinterpret_cast<float*>(smem + kOffArena + w * kArenaBytes);  // m[8] l[8] o[8][128]
    const int g = lane >> 2, h0 = 2 * (lane & 3);  // this lane: dims 16 t + g (+ 8), heads h0, h0 + 1
    const float l0 = col_sum(A.l[0]), l1 = col_sum(A.l[1]);
    if (g == 0) {
      wst[h0] = h0 < G ? A.m[0] : kNegInf;
      wst[h0 + 1] = h0 + 1 < G ? A.m[1] : kNegInf;
      wst[8 + h0] = h0 < G ? l0 : 0.f;
      wst[8 + h0 + 1] = h0 + 1 < G ? l1 : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      wst[16 + h0 * kHeadDim + 16 * t + g] = A.o[t][0];
      wst[16 + (h0 + 1) * kHeadDim + 16 * t + g] = A.o[t][1];
      wst[16 + h0 * kHeadDim + 16 * t + g + 8] = A.o[t][2];
      wst[16 + (h0 + 1) * kHeadDim + 16 * t + g + 8] = A.o[t][3];
    }
  }
  __syncthreads();
  // this CTA's partial: m[8], l[8], then o[h][128] for the G heads only
  const int pstride = 16 + G * kHeadDim;  // floats (a multiple of 4: 16-byte aligned)
  float* mine = P.partials + (size_t(C.g) * P.cg + C.j) * pstride;
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
      mine[16 + h * kHeadDim + d] = O;
      if (d == 0) {
        mine[h] = M;
        mine[8 + h] = L;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    // release: the CTA's partial (stored by every thread before the barrier)
    // is visible before the count; acquire: the last CTA sees every partial
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(old) : "l"(&P.groups[C.g].done) : "memory");
    ms->is_last = (old == P.cg - 1);
  }
  __syncthreads();
  if (!ms->is_last) return;

  // ---- last CTA of this group: merge the partials, write the output --------
  // (the partials arrive by bulk copy, kMergeChunk CTAs per copy, so the
  // merge costs one global round trip per chunk; an online log-sum-exp
  // merge runs over the chunks)
  const int cg = P.cg;
  const float* parts = P.partials + size_t(C.g) * cg * pstride;
  const float* cbuf = reinterpret_cast<const float*>(smem);  // chunk of partials
  float* sc = reinterpret_cast<float*>(smem + kMergeChunk * sizeof(Partial));  // [32][8] scales
  float* MLa = sc + kMergeChunk * 8;  // running M[8], L[8], and this chunk's rescale a[8]
  const int d = tid & (kHeadDim - 1), hsel = tid >> 7;  // this thread: dim d of heads hsel + 2i
  float Oh[4] = {0.f, 0.f, 0.f, 0.f};
  if (tid < 8) {
    MLa[tid] = kNegInf;
    MLa[8 + tid] = 0.f;
  }
  for (int c0 = 0, ph = 0; c0 < cg; c0 += kMergeChunk, ph ^= 1) {
    const int nc = (cg - c0) < kMergeChunk ? (cg - c0) : kMergeChunk;
    __syncthreads();  // the previous chunk is consumed
    if (tid == 0) {
      fence_proxy_async_global();
      mbar_arrive_expect_tx(&ms->cmb_bar, uint32_t(nc * pstride * 4));
      bulk_g2s(smem, parts + size_t(c0) * pstride, uint32_t(nc * pstride * 4), &ms->cmb_bar);
    }
    // every thread takes every barrier of this loop, even after a timeout
    // parked: the warps resume as the copy completes (a polling loop that
    // backs off with sleeps can oversleep it)
    const bool landed = mbar_wait_parked(&ms->cmb_bar, uint32_t(ph), kMergeWaitNs);
    if (!landed && tid == 0) set_device_error(P.status, DEV_WAIT_TIMEOUT, 7);
    // warp h: log-sum-exp statistics of head h over the chunk's CTAs (lane =
    // CTA), one shuffle reduction each, and every CTA's rescale factor
    if (w < G) {
      const float m = (landed && lane < nc) ? cbuf[lane * pstride + w] : kNegInf;
      const float l = (landed && lane < nc) ? cbuf[lane * pstride + 8 + w] : 0.f;
      float mc = m;
#pragma unroll
      for (int o = 16; o; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kFull, mc, o));
      const float m_old = MLa[w];
      const float m_new = fmaxf(m_old, mc);
      const float s_j = (m_new == kNegInf) ? 0.f : exp2f(m - m_new);
      float lc = l * s_j;
#pragma unroll
      for (int o = 16; o; o >>= 1) lc += __shfl_xor_sync(kFull, lc, o);
      if (lane < kMergeChunk) sc[lane * 8 + w] = s_j;
      __syncwarp();
      if (lane == 0) {
        const float a = (m_new == kNegInf) ? 1.f : exp2f(m_old - m_new);  // 0 on the first chunk
        MLa[16 + w] = a;
        MLa[w] = m_new;
        MLa[8 + w] = MLa[8 + w] * a + lc;
      }
    }
    __syncthreads();
    // every thread: its outputs, rescaled, plus the chunk's weighted sums
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int h = hsel + 2 * i;
      if (h >= G) continue;
      float o0 = Oh[i] * MLa[16 + h], o1 = 0.f, o2 = 0.f, o3 = 0.f;
      int jj = 0;
      for (; jj + 4 <= nc; jj += 4) {
        o0 = fmaf(cbuf[(jj + 0) * pstride + 16 + h * kHeadDim + d], sc[(jj + 0) * 8 + h], o0);
        o1 = fmaf(cbuf[(jj + 1) * pstride + 16 + h * kHeadDim + d], sc[(jj + 1) * 8 + h], o1);
        o2 = fmaf(cbuf[(jj + 2) * pstride + 16 + h * kHeadDim + d], sc[(jj + 2) * 8 + h], o2);
        o3 = fmaf(cbuf[(jj + 3) * pstride + 16 + h * kHeadDim + d], sc[(jj + 3) * 8 + h], o3);
      }
      for (; jj < nc; ++jj)
        o0 = fmaf(cbuf[jj * pstride + 16 + h * kHeadDim + d], sc[jj * 8 + h], o0);
      Oh[i] = (o0 + o1) + (o2 + o3);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int h = hsel + 2 * i;
    if (h < G) {
      const float L = MLa[8 + h];
      const size_t row = MQ ? (size_t(C.b) * P.nq_all + h / P.hpg) * P.Hq + size_t(C.c) * P.hpg + h % P.hpg
                            : size_t(C.b) * P.Hq + size_t(C.c) * G + h;
      P.out[row * kHeadDim + d] = L > 0.f ? Oh[i] / L : 0.f;
      if (d == 0 && P.lse != nullptr) P.lse[row] = L > 0.f ? (MLa[h] + log2f(L)) * kLn2 : kNegInf;
    }
  }
  if (P.fused && P.expanded_out != nullptr) {
    // the CTAs' ascending lists, one after the other
    int* pre = reinterpret_cast<int*>(MLa + 24);  // [cg + 1]
    __syncthreads();
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
      int sk0, sk1;
      span_range(jj, cg, C.n_sp, sk0, sk1);
      const int cnt = pre[jj + 1] - pre[jj];
      for (int i = lane; i < cnt; i += 32)
        P.expanded_out[C.gs + pre[jj] + i] = __ldcg(P.cta_list + C.gs + sk0 + i);
    }
    if (tid == 0 && P.n_expanded_out != nullptr) P.n_expanded_out[C.g] = pre[cg];
  }
  __syncthreads();
  if (tid == 0) {
    P.groups[C.g].done = 0;
    P.groups[C.g].full_next = 0;
  }
}

// grid: (cg, Hkv, B); block: 8 warps, each its own producer and consumer
template <int KS, bool MQ>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned (TMA's 128-byte swizzle), by pointer arithmetic on the
  // shared array itself: the compiler keeps every access through `smem` in
  // the shared window (32-bit addresses, shared loads and stores) instead of
  // generic 64-bit ones, as it would after a round trip through an integer
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  SmemMisc* ms = reinterpret_cast<SmemMisc*>(smem + kOffMisc);
  // fused mode: lane (r = lane / 4, dq = lane % 4) of warp w keeps the
  // 16-byte chunks c = dq + 4 i (i = 0..7) of W_r row 8w + r in registers
  // for the projection y = W_r q.  They are requested first, so their round
  // trip overlaps the set-up below and the wait for the query (the caller
  // allows W_r to be read before that wait).
  float4 wr[8];
  if (P.fused) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const float4* wrow = reinterpret_cast<const float4*>(
        P.W_r + (size_t(blockIdx.y) * kRouteDim + 8 * w + (lane >> 2)) * kHeadDim);
#pragma unroll
    for (int i = 0; i < 8; ++i) wr[i] = ldg_nc_early(wrow + (lane & 3) + 4 * i);
  }
  if (threadIdx.x < kWarps) {
    WarpQ& Q = ms->wq[threadIdx.x];
    Q = WarpQ{};
    Q.ok = 1;
  }
  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w)
      for (int s = 0; s < kSlots; ++s) mbar_init(&ms->bar[w][s], 1);
    mbar_init(&ms->cmb_bar, 1);
    ms->n_front = 0;
    ms->n_back = 0;
    ms->rec_next = 0;
    ms->fixed_next = 0;
    ms->is_last = 0;
    for (int p = 0; p < kMaxRoutePages; ++p) ms->pmask[p] = 0u;
    Ctx& C = ms->ctx;
    C.j = blockIdx.x;
    C.c = blockIdx.y;
    C.b = blockIdx.z;
    C.g = C.b * P.Hkv + C.c;
    C.gs = (long long)C.g * P.max_spans;
    C.bs = (long long)C.b * P.max_spans;
    C.n_sp = P.n_spans[C.b];
    C.n_full = P.n_sink + C.n_sp + (P.n_tail != nullptr ? P.n_tail[C.b] : P.n_recent);
    span_range(C.j, P.cg, C.n_sp, C.k0, C.k1);
    C.n_fp = (C.n_full + kFullRows - 1) / kFullRows;
    C.own0 = kStaticPages * C.j;
    const int own = C.n_fp - C.own0;
    C.n_own = own < 0 ? 0 : (own > kStaticPages ? kStaticPages : own);
    C.pool0 = kStaticPages * P.cg;
    C.n_fixed = C.n_own + (C.k1 - C.k0 + kRows - 1) / kRows;
    C.n_rp = P.fused ? (C.k1 - C.k0 + kRouteSpans - 1) / kRouteSpans : 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  run_decode<KS, MQ>(smem, ms, P, wr);
}

}  // namespace sekv
