// Producer warp of the decode kernel: streams pages into the consumer warps'
// rings (lane 0 issues; the whole warp helps in the expanded phase).
//
// Every page after the routing barrier goes to whichever consumer warp has a
// free slot first, so a warp busy with a heavy page never holds up the others.
#pragma once

#include "decode_attn.cuh"

namespace sekv {

// Issue state, passed by value (it stays in registers across the calls).
struct ProdState {
  uint32_t rs;        // per warp w: bit 2w = next slot (0/1), bit 2w+1 = its phase
  uint32_t filled;    // per slot: a page was ever issued into it
  uint32_t last_par;  // per slot: phase of the last page issued into it
  int rr;             // warp tried first by the next pick
  int ok;             // no wait has timed out
  uint32_t spm;       // bit w: warp w is consuming a record larger than a page
};

__device__ __forceinline__ int ring_slot(const ProdState& S, int w) {
  return w * kSlotsPerWarp + int((S.rs >> (2 * w)) & 1u);
}
__device__ __forceinline__ uint32_t ring_phase(const ProdState& S, int w) {
  return (S.rs >> (2 * w + 1)) & 1u;
}

// Bit w set iff warp w's next slot is free (the four tests overlap).
__device__ __forceinline__ uint32_t free_warps(SmemMisc* ms, const ProdState& S) {
  const uint32_t e0 = smem_u32(&ms->empty[0]);
  return mbar_test4(e0 + 8u * ring_slot(S, 0), e0 + 8u * ring_slot(S, 1),
                    e0 + 8u * ring_slot(S, 2), e0 + 8u * ring_slot(S, 3), ring_phase(S, 0) ^ 1u,
                    ring_phase(S, 1) ^ 1u, ring_phase(S, 2) ^ 1u, ring_phase(S, 3) ^ 1u);
}

// Warps whose record larger than a page is still in progress (acquire: a
// cleared flag comes after that warp's last release of its ring slots).
__device__ __forceinline__ uint32_t busy_warps(SmemMisc* ms) {
  uint32_t m = 0;
#pragma unroll
  for (int x = 0; x < kConsumerWarps; ++x) m |= ld_acquire_cta(&ms->sp_busy[x]) ? (1u << x) : 0u;
  return m;
}

// First warp (from S.rr on, never one still consuming a record larger than a
// page) whose next slot is free; bounded.
__device__ __forceinline__ int pick_warp(uint8_t* smem, SmemMisc* ms, ProdState& S,
                                         const DecodeParams& P) {
  static_assert(kConsumerWarps == 4, "four consumer warps");
  int w = 0;
  for (uint32_t it = 0;; ++it) {
    if (S.spm) S.spm &= busy_warps(ms);
    // a warp consuming a large record has its ring slots ahead in use
    const uint32_t fm = free_warps(ms, S) & ~S.spm;
    if (fm) {
      // the first free warp from S.rr on
      const uint32_t rot = ((fm | (fm << 4)) >> S.rr) & 0xFu;
      w = (S.rr + __ffs(rot) - 1) & 3;
      break;
    }
    if (it >= kWaitLimit || !S.ok) {
      set_device_error(P.status, DEV_WAIT_TIMEOUT, 6);
      S.ok = 0;
      return 0;
    }
    if (it > 64) __nanosleep(32);
  }
  S.rr = (w + 1) & (kConsumerWarps - 1);
  return w;
}

// Bounded wait for warp w's next slot (pages that must go to that warp).
__device__ __forceinline__ bool wait_warp(SmemMisc* ms, ProdState& S, int w, int32_t* status) {
  if (!mbar_wait(&ms->empty[ring_slot(S, w)], ring_phase(S, w) ^ 1u, kWaitLimit)) {
    set_device_error(status, DEV_WAIT_TIMEOUT, 1);
    S.ok = 0;
    return false;
  }
  return true;
}

// Warp w's next slot, known free: publish the descriptor, then arm the full
// barrier, so that the consumer's acquire on the barrier covers it.
__device__ __forceinline__ int arm_page(SmemMisc* ms, const ProdState& S, int w,
                                        const PageDesc& d, uint32_t bytes) {
  const int slot = ring_slot(S, w);
  ms->desc[slot] = d;
  mbar_arrive_expect_tx(&ms->full[slot], bytes);
  return slot;
}

__device__ __forceinline__ void commit_page(ProdState& S, int w, int slot) {
  S.filled |= 1u << slot;
  S.last_par = (S.last_par & ~(1u << slot)) | (ring_phase(S, w) << slot);
  // advance warp w's ring: the slot bit flips, the phase flips after slot 1
  const uint32_t v = (S.rs >> (2 * w)) & 3u;
  const uint32_t nv = (v ^ 1u) ^ ((v & 1u) << 1);
  S.rs = (S.rs & ~(3u << (2 * w))) | (nv << (2 * w));
}

// Small records staged for the next multi-record page: lane i holds record
// i (its source offset and table entry); n and bytes are the same in every lane.
struct Batch {
  int n, bytes;
  long long src;
  RecInfo ri;
};

// The staged records as one page.  Called by the whole warp: lane 0 picks
// the warp and arms the barrier, every staged lane writes its table entry
// and issues its own copy.
__device__ __forceinline__ void flush_batch(uint8_t* smem, SmemMisc* ms, ProdState& S,
                                            const DecodeParams& P, Batch& B) {
  const int lane = threadIdx.x & 31;
  if (B.n == 0 || !S.ok) return;
  int slot = 0;
  if (lane == 0) {
    const int w = pick_warp(smem, ms, S, P);
    if (S.ok) {
      slot = ring_slot(S, w);
      PageDesc d{};
      d.type = PG_EXPM;
      d.n = B.n;
      ms->desc[slot] = d;
      commit_page(S, w, slot);  // ring state only: the barrier is armed below
    }
  }
  S.ok = __shfl_sync(0xffffffffu, S.ok, 0);
  slot = __shfl_sync(0xffffffffu, slot, 0);
  if (S.ok) {
    if (lane < B.n) ms->rec[slot][lane] = B.ri;
    __syncwarp();
    // the descriptor and the table are published by this arrive (release)
    if (lane == 0) mbar_arrive_expect_tx(&ms->full[slot], uint32_t(B.bytes));
    __syncwarp();
    if (lane < B.n)
      bulk_g2s_hint(slot_ptr(smem, slot) + B.ri.off, P.store + B.src,
                    uint32_t(record_bytes(B.ri.b, B.ri.rk, B.ri.rv)), &ms->full[slot],
                    policy_evict_first());
  }
  B.n = 0;
  B.bytes = 0;
}

// A record larger than a page goes to one warp as several pages: its key
// part, its U rows in tiles, its value part (the partial state of the span
// stays in that warp's registers).  The producer hands over part 0 and
// counts all the parts into that warp's ring; the warp loads each further
// part into its other slot itself as it starts on the one before, so the
// parts follow each other at the warp's own pace.
__device__ __forceinline__ ProdState start_split(uint8_t* smem, SmemMisc* ms, ProdState S,
                                                 const DecodeParams& P, int b, int rank,
                                                 long long off) {
  const int w = pick_warp(smem, ms, S, P);
  if (!S.ok) return S;
  const int rK = rank & 0xFFFF, rV = (rank >> 16) & 0xFFFF;
  // Until the warp clears its flag the producer's view of its ring runs
  // ahead of the barriers (all parts counted in), and a one-bit parity test
  // would take a phase two back for the awaited one: its slots go untested.
  ms->sp_busy[w] = 1;
  const int slot = ring_slot(S, w);
  issue_split_part(smem, ms, P, slot, 0, b, rK, rV, off);
  const int np = split_nparts(b, rK, rV);
  for (int k = 0; k < np; ++k) commit_page(S, w, ring_slot(S, w));
  S.spm |= 1u << w;
  return S;
}

// Every large record handed over has been consumed (bounded wait).
__device__ __forceinline__ ProdState finish_splits(SmemMisc* ms, ProdState S,
                                                   const DecodeParams& P) {
  for (uint32_t it = 0; S.spm && S.ok; ++it) {
    S.spm &= busy_warps(ms);
    if (it >= kWaitLimit) {
      set_device_error(P.status, DEV_WAIT_TIMEOUT, 8);
      S.ok = 0;
    }
    if (it > 64) __nanosleep(32);
  }
  return S;
}

// Fixed page t of this CTA: full-resolution rows first, then summary rows,
// 32 per page, to the first warp with a free slot.
__device__ __forceinline__ ProdState issue_fixed(uint8_t* smem, SmemMisc* ms, ProdState S,
                                              const DecodeParams& P, int t, int nfp, int f0,
                                              int f1, int k0, int k1, int g) {
  const int w = pick_warp(smem, ms, S, P);
  if (!S.ok) return S;
  PageDesc d{};
  const bool full = t < nfp;
  const int a = full ? f0 + kTileRows * t : k0 + kTileRows * (t - nfp);
  const int e = full ? f1 : k1;
  d.type = full ? PG_FULL : PG_SUM;
  d.n = (e - a) < kTileRows ? (e - a) : kTileRows;
  d.a = a;
  const int slot = arm_page(ms, S, w, d, 4 * kBoxBytes);
  uint8_t* pg = slot_ptr(smem, slot);
  const CUtensorMap* tk = full ? &P.tm_kfull : &P.tm_ksum;
  const CUtensorMap* tv = full ? &P.tm_vfull : &P.tm_vsum;
  const uint64_t pol = policy_evict_first();
  tma_g2s_4d_hint(pg, tk, 0, a, 0, g, &ms->full[slot], pol);                  // both halves of K
  tma_g2s_4d_hint(pg + 2 * kBoxBytes, tv, 0, a, 0, g, &ms->full[slot], pol);  // both halves of V
  commit_page(S, w, slot);
  return S;
}

// Inclusive warp scan of a 64-bit value.
__device__ __forceinline__ long long warp_incl_scan(long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

static __device__ void producer_warp(uint8_t* smem, SmemMisc* ms, const DecodeParams& P, int g, int j,
                              int b, int c) {
  const int lane = threadIdx.x & 31;
  const int n_sp = P.n_spans[b];
  const int n_full = P.n_sink + n_sp + P.n_recent;
  int f0, f1, k0, k1;
  fixed_range(j, P.cg, n_full, n_sp, P.fused, f0, f1, k0, k1);
  const int nfp = (f1 - f0 + kTileRows - 1) / kTileRows;
  const int nfixed = nfp + (k1 - k0 + kTileRows - 1) / kTileRows;
  ProdState S{0u, 0u, 0u, 0, 1, 0u};
  const size_t gs = size_t(g) * P.max_spans;
  int t_fixed = 0;  // fixed pages issued so far

  // list mode reads what the preparation kernel wrote: wait for it first
  if (!P.fused) pdl_wait();
  if (lane == 0) {
    prefetch_tmap(&P.tm_kfull);
    prefetch_tmap(&P.tm_vfull);
    prefetch_tmap(&P.tm_ksum);
    prefetch_tmap(&P.tm_vsum);
    PageDesc d{};
    if (P.fused) {
      prefetch_tmap(&P.tm_sroute);
      // routing weights of this KV head in one copy (four 128B-swizzled blocks
      // of 64 rows x 32 floats); every CTA of the head reads them: kept in L2
      mbar_arrive_expect_tx(&ms->wr_bar, kRouteDim * kHeadDim * 4);
      tma_g2s_4d_hint(smem + kOffWr, &P.tm_wr, 0, 0, 0, c, &ms->wr_bar, policy_evict_last());
      // routing pages, 64 spans each
      const uint64_t pol = policy_evict_first();
      for (int k = k0, p = 0; S.ok && k < k1; k += kRouteSpans, ++p) {
        const int n = (k1 - k) < kRouteSpans ? (k1 - k) : kRouteSpans;
        d.type = PG_ROUTE; d.n = n; d.a = k; d.flag = p;
        const int w = pick_warp(smem, ms, S, P);
        if (!S.ok) break;
        // the routing summaries of 64 spans, both halves of each row (the
        // consumer reads the spans' metadata from global memory itself)
        const int slot = arm_page(ms, S, w, d, 2 * 8192);
        tma_g2s_4d_hint(slot_ptr(smem, slot), &P.tm_sroute, 0, k, 0, g, &ms->full[slot], pol);
        commit_page(S, w, slot);
      }
    } else if (k1 > k0) {
      const int n = k1 - k0;
      const uint32_t bytes = uint32_t(pad16(2 * int64_t(n)));
      d.type = PG_INFO; d.n = n; d.a = k0;
      if (wait_warp(ms, S, 0, P.status)) {
        const int slot = arm_page(ms, S, 0, d, bytes);
        bulk_g2s(slot_ptr(smem, slot), P.info + gs + k0, bytes, &ms->full[slot]);
        commit_page(S, 0, slot);
      }
    }
    // every warp passes the routing barrier at this page
    for (int w = 0; S.ok && w < kConsumerWarps; ++w) {
      d = PageDesc{};
      d.type = PG_SYNC;
      if (wait_warp(ms, S, w, P.status)) commit_page(S, w, arm_page(ms, S, w, d, 0));
    }
  }

  // Until every CTA of this KV head has published its expanded spans, keep
  // the warps busy with fixed pages (at most three quarters of them: the
  // rest balance the tail).
  pdl_wait();
  if (lane == 0 && S.ok) {
    const int part = (3 * nfixed + 3) / 4;
    while (S.ok && t_fixed < part) {
      if (P.fused && ld_acquire(&P.groups[g].published) >= P.cg) break;
      S = issue_fixed(smem, ms, S, P, t_fixed, nfp, f0, f1, k0, k1, g);
      ++t_fixed;
    }
  }
  S.ok = __shfl_sync(0xffffffffu, S.ok, 0);
  t_fixed = __shfl_sync(0xffffffffu, t_fixed, 0);

  // expanded spans: wait until every CTA of this KV head has published,
  // then take the entries whose byte offset falls in this CTA's share.
  if (S.ok && P.fused) {
    int pub = 0;
    if (lane == 0) {
      uint32_t it = 0;
      while ((pub = ld_acquire(&P.groups[g].published)) < P.cg && it < kSpinLimit) {
        ++it;
        __nanosleep(64);
      }
      if (pub < P.cg) set_device_error(P.status, DEV_WAIT_TIMEOUT, 2);
    }
    pub = __shfl_sync(0xffffffffu, pub, 0);
    if (pub < P.cg) S.ok = 0;
  }
  Batch B{0, 0, 0, RecInfo{}};  // staged small records
  if (S.ok) {
    const int cg = P.cg;
    // round trip 1: expanded-span counts and bytes of every CTA, prefixed
    {
      long long carry = 0;
      int ncarry = 0;
      for (int j0 = 0; j0 < cg; j0 += 32) {
        const int jj = j0 + lane;
        const long long v =
            jj < cg ? __ldcg(reinterpret_cast<const long long*>(P.cta_bytes) + size_t(g) * cg + jj)
                    : 0;
        const int cn = jj < cg ? __ldcg(P.cta_n + size_t(g) * cg + jj) : 0;
        const long long inc = warp_incl_scan(v);
        const long long incn = warp_incl_scan(cn);
        if (jj < cg) {
          ms->pre_b[jj] = carry + inc - v;
          ms->pre_n[jj] = ncarry + int(incn) - cn;
        }
        carry += __shfl_sync(0xffffffffu, inc, 31);
        ncarry += int(__shfl_sync(0xffffffffu, incn, 31));
      }
      if (lane == 0) {
        ms->pre_b[cg] = carry;
        ms->pre_n[cg] = ncarry;
      }
      __syncwarp();
    }
    const long long Tb = ms->pre_b[cg];
    const long long lo = byte_split(Tb, j, cg), hi = byte_split(Tb, j + 1, cg);
    // lanes hold candidate entries in byte order; those that start in
    // [lo, hi) go into the current batch, or out as split records (every
    // lane follows the batch; lane 0 alone issues)
    auto offer = [&](bool mine, const ExpEntry& en) {
      uint32_t bal = __ballot_sync(0xffffffffu, mine);
      while (bal && S.ok) {
        const int src = __ffs(bal) - 1;
        bal &= bal - 1;
        const int body = __shfl_sync(0xffffffffu, en.body, src);
        const int rank = __shfl_sync(0xffffffffu, en.rank, src);
        const long long off = __shfl_sync(0xffffffffu, en.off, src);
        const int xr = rank & 0xFFFF, xv = (rank >> 16) & 0xFFFF;
        const int sz = int(record_bytes(body, xr, xv));
        if (xr > P.rank_lim || xv > P.rank_lim) {
          if (lane == 0) set_device_error(P.status, DEV_BAD_RANK, xr > xv ? xr : xv);  // skipped
        } else if (sz > kPageData) {
          if (lane == 0) S = start_split(smem, ms, S, P, body, rank, off);
        } else {
          if (B.n == kMaxRecPerPage || B.bytes + sz > kPageData) flush_batch(smem, ms, S, P, B);
          if (lane == B.n) {
            B.src = off;
            B.ri = RecInfo{B.bytes, body, xr, xv};
          }
          B.bytes += sz;
          ++B.n;
        }
        S.ok = __shfl_sync(0xffffffffu, S.ok, 0);
      }
    };
    for (int jj = 0; jj < cg && S.ok; ++jj) {
      const int cnt = ms->pre_n[jj + 1] - ms->pre_n[jj];
      if (cnt == 0 || ms->pre_b[jj + 1] <= lo) continue;
      if (ms->pre_b[jj] >= hi) break;
      if (!P.fused) {
        // list mode: one compact sublist with per-entry byte offsets
        const ExpEntry* base = P.entries + gs;
        for (int e0 = 0; e0 < cnt && S.ok; e0 += 32) {
          ExpEntry en{};
          bool mine = false;
          if (e0 + lane < cnt) {
            const int4* src = reinterpret_cast<const int4*>(base + e0 + lane);
            const int4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
            en.k = v0.x; en.body = v0.y; en.rank = v0.z;
            en.off = (long long)(uint32_t(v1.x)) | ((long long)v1.y << 32);
            const long long cum = (long long)(uint32_t(v1.z)) | ((long long)v1.w << 32);
            const long long st = ms->pre_b[jj] + cum;
            mine = st >= lo && st < hi && en.body > 0;
          }
          offer(mine, en);
        }
        continue;
      }
      // fused mode, round trip 2: CTA jj's routing pages (one per lane)
      int a0, a1, sk0, sk1;
      fixed_range(jj, cg, n_full, n_sp, 1, a0, a1, sk0, sk1);
      const int npj = (sk1 - sk0 + kRouteSpans - 1) / kRouteSpans;
      const size_t pb = (size_t(g) * cg + jj) * kMaxRoutePages;
      const long long pbytes =
          lane < npj ? __ldcg(reinterpret_cast<const long long*>(P.pbytes) + pb + lane) : 0;
      const unsigned long long pmask =
          lane < npj ? __ldcg(reinterpret_cast<const unsigned long long*>(P.pmask) + pb + lane)
                     : 0ull;
      const long long pstart = ms->pre_b[jj] + warp_incl_scan(pbytes) - pbytes;
      const bool hit = lane < npj && pbytes > 0 && pstart < hi && pstart + pbytes > lo;
      const int cntp = hit ? __popcll(pmask) : 0;
      const int cincl = int(warp_incl_scan(cntp));
      const int cpre = cincl - cntp;
      const int E = __shfl_sync(0xffffffffu, cincl, 31);
      // round trip 3: the entries of the hit pages, flattened over the lanes
      for (int f0 = 0; f0 < E && S.ok; f0 += 32) {
        const int f = f0 + lane;
        int pl = 0;  // last page whose entry prefix is <= f
#pragma unroll
        for (int step = 16; step; step >>= 1) {
          const int v = __shfl_sync(0xffffffffu, cpre, (pl + step) & 31);
          if (pl + step < 32 && v <= f) pl += step;
        }
        const int i = f - __shfl_sync(0xffffffffu, cpre, pl);
        const long long pst = __shfl_sync(0xffffffffu, pstart, pl);
        ExpEntry en{};
        bool mine = false;
        if (f < E) {
          const int4* src = reinterpret_cast<const int4*>(P.entries + gs + sk0 +
                                                          kRouteSpans * pl + i);
          const int4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
          en.k = v0.x; en.body = v0.y; en.rank = v0.z;
          en.off = (long long)(uint32_t(v1.x)) | ((long long)v1.y << 32);
          const long long cum = (long long)(uint32_t(v1.z)) | ((long long)v1.w << 32);
          const long long st = pst + cum;
          mine = st >= lo && st < hi;
        }
        offer(mine, en);
      }
    }
  }
  flush_batch(smem, ms, S, P, B);
  if (lane == 0) {
    // the remaining fixed pages, to whichever warp frees a slot first
    while (S.ok && t_fixed < nfixed) {
      S = issue_fixed(smem, ms, S, P, t_fixed, nfp, f0, f1, k0, k1, g);
      ++t_fixed;
    }
    S = finish_splits(ms, S, P);
    // every consumer warp ends with an END page
    for (int w = 0; w < kConsumerWarps; ++w) {
      PageDesc d{};
      d.type = PG_END;
      ProdState S2 = S;
      S2.ok = 1;
      if (wait_warp(ms, S2, w, P.status)) commit_page(S2, w, arm_page(ms, S2, w, d, 0));
      S.rs = S2.rs;
      S.filled = S2.filled;
      S.last_par = S2.last_par;
    }
    // drain: every issued copy has landed before the CTA may exit
    for (int s = 0; s < kSlots; ++s)
      if (((S.filled >> s) & 1u) &&
          !mbar_wait(&ms->full[s], (S.last_par >> s) & 1u, kWaitLimit))
        set_device_error(P.status, DEV_WAIT_TIMEOUT, 3);
  }
}

}  // namespace sekv
