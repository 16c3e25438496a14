// Producer warp of the decode kernel: streams pages into the ring.
#pragma once

#include "decode_attn.cuh"

namespace sekv {

// Issue the pages of one expanded span.  A record that fits a page goes in
// one copy; a larger one as its key part, its U rows in tiles, its value part.
__device__ __forceinline__ bool issue_expanded(uint8_t* smem, SmemMisc* ms, Ring& r,
                                               const DecodeParams& P, const ExpEntry& e,
                                               uint32_t* last_par, bool* filled) {
  bool ok = true;
  const int b = e.body, rK = e.rank & 0xFFFF, rV = (e.rank >> 16) & 0xFFFF;
  const uint8_t* rec = P.store + e.off;
  const RecordLayout L = record_layout(b, rK, rV);
  PageDesc d{};
  d.type = PG_EXP;
  d.rk = rK;
  d.rv = rV;
  if (L.total <= kPageData) {
    d.n = b; d.a = 0;
    d.off_a = 0; d.off_uk = int(L.uk); d.off_uv = int(L.uv); d.off_b = int(L.vpart);
    uint8_t* pg = push_page(smem, ms, r, d, uint32_t(L.total), P.status, ok);
    if (!ok) return false;
    bulk_g2s(pg, rec, uint32_t(L.total), &ms->full[r.slot]);
    filled[r.slot] = true;
    last_par[r.slot] = r.phase;
    advance(r);
    return true;
  }
  // key part
  d.n = 0; d.a = 0; d.off_a = 0; d.off_uk = 0; d.off_uv = 0; d.off_b = -1;
  {
    uint8_t* pg = push_page(smem, ms, r, d, uint32_t(L.uk), P.status, ok);
    if (!ok) return false;
    bulk_g2s(pg, rec, uint32_t(L.uk), &ms->full[r.slot]);
    filled[r.slot] = true;
    last_par[r.slot] = r.phase;
    advance(r);
  }
  // U rows: [i0, i0 + n) of U_K at +0 and of U_V at +16384
  const int rmax = r8(rK) > r8(rV) ? r8(rK) : r8(rV);
  int rows = rmax > 0 ? (16384 / (2 * rmax)) & ~15 : 512;
  if (rows > 512) rows = 512;
  for (int i0 = 0; i0 < b; i0 += rows) {
    const int n = (b - i0) < rows ? (b - i0) : rows;
    const uint32_t bk = uint32_t(2 * n * r8(rK)), bv = uint32_t(2 * n * r8(rV));
    d.n = n; d.a = i0; d.off_a = -1; d.off_uk = 0; d.off_uv = 16384; d.off_b = -1;
    uint8_t* pg = push_page(smem, ms, r, d, bk + bv, P.status, ok);
    if (!ok) return false;
    if (bk) bulk_g2s(pg, rec + L.uk + 2 * int64_t(i0) * r8(rK), bk, &ms->full[r.slot]);
    if (bv) bulk_g2s(pg + 16384, rec + L.uv + 2 * int64_t(i0) * r8(rV), bv, &ms->full[r.slot]);
    filled[r.slot] = true;
    last_par[r.slot] = r.phase;
    advance(r);
  }
  // value part
  {
    const uint32_t bytes = uint32_t(L.total - L.vpart);
    d.n = 0; d.a = 0; d.off_a = -1; d.off_b = 0;
    uint8_t* pg = push_page(smem, ms, r, d, bytes, P.status, ok);
    if (!ok) return false;
    if (bytes) bulk_g2s(pg, rec + L.vpart, bytes, &ms->full[r.slot]);
    filled[r.slot] = true;
    last_par[r.slot] = r.phase;
    advance(r);
  }
  return true;
}

// Small records waiting to be packed into one page (producer lane 0).
struct Batch {
  int n = 0;
  int64_t bytes = 0;
  int64_t src[kMaxRecPerPage];
  RecInfo tab[kMaxRecPerPage];
};

__device__ __forceinline__ bool flush_batch(uint8_t* smem, SmemMisc* ms, Ring& r,
                                            const DecodeParams& P, Batch& bat,
                                            uint32_t* last_par, bool* filled) {
  if (bat.n == 0) return true;
  bool ok = true;
  PageDesc d{};
  d.type = PG_EXPM;
  d.n = bat.n;
  uint8_t* pg = push_page(smem, ms, r, d, uint32_t(bat.bytes), P.status, ok, bat.tab, bat.n);
  if (!ok) return false;
  for (int i = 0; i < bat.n; ++i) {
    const int64_t sz = record_bytes(bat.tab[i].b, bat.tab[i].rk, bat.tab[i].rv);
    bulk_g2s(pg + bat.tab[i].off, P.store + bat.src[i], uint32_t(sz), &ms->full[r.slot]);
  }
  filled[r.slot] = true;
  last_par[r.slot] = r.phase;
  advance(r);
  bat.n = 0;
  bat.bytes = 0;
  return true;
}

__device__ void producer_warp(uint8_t* smem, SmemMisc* ms, const DecodeParams& P, int g, int j,
                              int b, int c) {
  const int lane = threadIdx.x & 31;
  const int n_sp = P.n_spans[b];
  const int n_full = P.n_sink + n_sp + P.n_recent;
  int f0, f1, k0, k1;
  fixed_range(j, P.cg, n_full, n_sp, P.fused, f0, f1, k0, k1);
  Ring r;
  uint32_t last_par[kPages];
  bool filled[kPages];
#pragma unroll
  for (int s = 0; s < kPages; ++s) { filled[s] = false; last_par[s] = 0; }
  bool ok = true;
  const size_t gs = size_t(g) * P.max_spans;
  Batch bat;

  // list mode reads what the preparation kernel wrote: wait for it first
  if (!P.fused) pdl_wait();
  if (lane == 0) {
    prefetch_tmap(&P.tm_kfull);
    prefetch_tmap(&P.tm_vfull);
    prefetch_tmap(&P.tm_ksum);
    prefetch_tmap(&P.tm_vsum);
    if (P.fused) {
      prefetch_tmap(&P.tm_sroute);
      // routing weights of this KV head, rows padded to kWrStride bytes
      mbar_arrive_expect_tx(&ms->wr_bar, kRouteDim * kHeadDim * 4);
      for (int row = 0; row < kRouteDim; ++row)
        bulk_g2s(smem + kOffWr + row * kWrStride,
                 P.W_r + (size_t(c) * kRouteDim + row) * kHeadDim, kHeadDim * 4, &ms->wr_bar);
    }
    PageDesc d{};
    // 1. routing pages (fused) or the span-info page (list mode)
    if (P.fused) {
      int k = k0;
      do {
        const int n = (k1 - k) < kRouteSpans ? (k1 - k) : kRouteSpans;
        d.type = PG_ROUTE; d.n = n; d.a = k; d.flag = (k + n >= k1);
        const int nb = (n + 63) / 64;  // row boxes of 64 spans
        const uint32_t n4 = uint32_t((n + 3) & ~3);
        const uint32_t n2 = uint32_t((n + 1) & ~1);
        const uint32_t bytes = n > 0 ? nb * 2 * 8192 + n4 * 4 * 2 + n2 * 8 : 0;
        uint8_t* pg = push_page(smem, ms, r, d, bytes, P.status, ok);
        if (!ok) break;
        if (n > 0) {
          for (int rb = 0; rb < nb; ++rb)
            for (int cb = 0; cb < 2; ++cb)
              tma_g2s_3d(pg + (rb * 2 + cb) * 8192, &P.tm_sroute, cb * 32, k + rb * 64, g,
                         &ms->full[r.slot]);
          bulk_g2s(pg + kAuxBody, P.body_len + size_t(b) * P.max_spans + k, n4 * 4,
                   &ms->full[r.slot]);
          bulk_g2s(pg + kAuxRank, P.rec_rank + gs + k, n4 * 4, &ms->full[r.slot]);
          bulk_g2s(pg + kAuxOff, P.rec_off + gs + k, n2 * 8, &ms->full[r.slot]);
        }
        filled[r.slot] = true; last_par[r.slot] = r.phase;
        advance(r);
        k += n;
      } while (k < k1);
    } else if (ok) {
      const int n = k1 - k0;
      const uint32_t bytes = uint32_t(pad16(2 * int64_t(n)));
      d.type = PG_INFO; d.n = n; d.a = k0;
      uint8_t* pg = push_page(smem, ms, r, d, bytes, P.status, ok);
      if (ok) {
        if (bytes) bulk_g2s(pg, P.info + gs + k0, bytes, &ms->full[r.slot]);
        filled[r.slot] = true; last_par[r.slot] = r.phase;
        advance(r);
      }
    }
    // 2. full-resolution rows
    for (int f = f0; ok && f < f1; f += kTileRows) {
      const int n = (f1 - f) < kTileRows ? (f1 - f) : kTileRows;
      d.type = PG_FULL; d.n = n; d.a = f;
      uint8_t* pg = push_page(smem, ms, r, d, 4 * 8192, P.status, ok);
      if (!ok) break;
      tma_g2s_3d(pg, &P.tm_kfull, 0, f, g, &ms->full[r.slot]);
      tma_g2s_3d(pg + 8192, &P.tm_kfull, 64, f, g, &ms->full[r.slot]);
      tma_g2s_3d(pg + 16384, &P.tm_vfull, 0, f, g, &ms->full[r.slot]);
      tma_g2s_3d(pg + 24576, &P.tm_vfull, 64, f, g, &ms->full[r.slot]);
      filled[r.slot] = true; last_par[r.slot] = r.phase;
      advance(r);
    }
    // 3. summary rows of the span range
    for (int k = k0; ok && k < k1; k += kTileRows) {
      const int n = (k1 - k) < kTileRows ? (k1 - k) : kTileRows;
      d.type = PG_SUM; d.n = n; d.a = k;
      uint8_t* pg = push_page(smem, ms, r, d, 4 * 8192, P.status, ok);
      if (!ok) break;
      tma_g2s_3d(pg, &P.tm_ksum, 0, k, g, &ms->full[r.slot]);
      tma_g2s_3d(pg + 8192, &P.tm_ksum, 64, k, g, &ms->full[r.slot]);
      tma_g2s_3d(pg + 16384, &P.tm_vsum, 0, k, g, &ms->full[r.slot]);
      tma_g2s_3d(pg + 24576, &P.tm_vsum, 64, k, g, &ms->full[r.slot]);
      filled[r.slot] = true; last_par[r.slot] = r.phase;
      advance(r);
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);

  // 4. expanded spans: wait until every CTA of this KV head has published,
  // then take the entries whose byte offset falls in this CTA's share.
  pdl_wait();
  if (ok) {
    if (P.fused) {
      int pub = 0;
      if (lane == 0) {
        uint32_t it = 0;
        while ((pub = ld_acquire(&P.groups[g].published)) < P.cg && it < kSpinLimit) {
          ++it;
          __nanosleep(128);
        }
        if (pub < P.cg) set_device_error(P.status, DEV_WAIT_TIMEOUT, 2);
      }
      pub = __shfl_sync(0xffffffffu, pub, 0);
      if (pub < P.cg) ok = false;
    }
  }
  if (ok) {
    const int cg = P.cg;
    // per-CTA entry counts and byte totals -> exclusive prefixes in smem
    for (int jj = lane; jj < cg; jj += 32) {
      ms->pre_n[jj + 1] = __ldcg(P.cta_n + size_t(g) * cg + jj);
      ms->pre_b[jj + 1] = __ldcg(reinterpret_cast<const long long*>(P.cta_bytes) + size_t(g) * cg + jj);
    }
    __syncwarp();
    if (lane == 0) {
      ms->pre_n[0] = 0;
      ms->pre_b[0] = 0;
      for (int jj = 1; jj <= cg; ++jj) {
        ms->pre_n[jj] += ms->pre_n[jj - 1];
        ms->pre_b[jj] += ms->pre_b[jj - 1];
      }
    }
    __syncwarp();
    const long long Tb = ms->pre_b[cg];
    const long long lo = Tb * j / cg, hi = Tb * (j + 1) / cg;
    // walk the sublists that can hold entries starting in [lo, hi)
    for (int jj = 0; jj < cg && ok; ++jj) {
      const int cnt = ms->pre_n[jj + 1] - ms->pre_n[jj];
      if (cnt == 0 || ms->pre_b[jj + 1] <= lo) continue;
      if (ms->pre_b[jj] >= hi) break;
      int sk0 = 0;
      if (P.fused) {
        int a0, a1, a2;
        fixed_range(jj, cg, n_full, n_sp, 1, a0, a1, sk0, a2);
      }
      const ExpEntry* base = P.entries + gs + sk0;
      for (int e0 = 0; e0 < cnt && ok; e0 += 32) {
        ExpEntry en{};
        bool mine = false;
        if (e0 + lane < cnt) {
          const int4* src = reinterpret_cast<const int4*>(base + e0 + lane);
          int4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
          en.k = v0.x; en.body = v0.y; en.rank = v0.z;
          en.off = (long long)(uint32_t(v1.x)) | ((long long)v1.y << 32);
          const long long cum = (long long)(uint32_t(v1.z)) | ((long long)v1.w << 32);
          const long long st = ms->pre_b[jj] + cum;
          mine = st >= lo && st < hi && en.body > 0;
        }
        uint32_t bal = __ballot_sync(0xffffffffu, mine);
        while (bal && ok) {
          const int src_lane = __ffs(bal) - 1;
          bal &= bal - 1;
          ExpEntry x;
          x.k = __shfl_sync(0xffffffffu, en.k, src_lane);
          x.body = __shfl_sync(0xffffffffu, en.body, src_lane);
          x.rank = __shfl_sync(0xffffffffu, en.rank, src_lane);
          x.off = __shfl_sync(0xffffffffu, en.off, src_lane);
          if (lane == 0) {
            const int xr = x.rank & 0xFFFF, xv = (x.rank >> 16) & 0xFFFF;
            const int64_t sz = record_bytes(x.body, xr, xv);
            if (sz > kPageData) {  // too big for a page: split path
              ok = flush_batch(smem, ms, r, P, bat, last_par, filled);
              if (ok) ok = issue_expanded(smem, ms, r, P, x, last_par, filled);
            } else {
              if (bat.n == kMaxRecPerPage || bat.bytes + sz > kPageData)
                ok = flush_batch(smem, ms, r, P, bat, last_par, filled);
              bat.src[bat.n] = x.off;
              bat.tab[bat.n] = RecInfo{int(bat.bytes), x.body, xr, xv};
              bat.bytes += sz;
              ++bat.n;
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
    }
  }
  if (lane == 0 && ok) ok = flush_batch(smem, ms, r, P, bat, last_par, filled);
  if (lane == 0) {
    PageDesc d{};
    d.type = PG_END;
    bool ok2 = true;
    push_page(smem, ms, r, d, 0, P.status, ok2);
    if (ok2) { filled[r.slot] = true; last_par[r.slot] = r.phase; advance(r); }
    // drain: every issued copy has landed before the CTA may exit
    for (int s = 0; s < kPages; ++s)
      if (filled[s] && !mbar_wait(&ms->full[s], last_par[s], kWaitLimit))
        set_device_error(P.status, DEV_WAIT_TIMEOUT, 3);
  }
}

}  // namespace sekv
