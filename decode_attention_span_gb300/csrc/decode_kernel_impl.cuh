// The decode kernel's body: routing pages, publication, the consumer warps
// and the kernel itself, a template on KS (rank k-steps of 16: ranks up to
// 16 KS).  Each KS is instantiated in a translation unit of its own.
#pragma once

#include "decode_consumer.cuh"
#include "decode_producer.cuh"

namespace sekv {

// Routing page (64 spans), processed by one warp: z_h = y_h . s_S in fp32
// FMAs, then two spans per lane for the bookkeeping.  A span expands
// iff its body is non-empty and some head of the group has z_h > theta_h.
// The page's expanded spans get compact entries from the page's first span
// ordinal on; the page keeps a bit mask of them and their record bytes.
__device__ __forceinline__ void consume_route(const uint8_t* page, const PageDesc& d, int k0,
                                              const DecodeParams& P, SmemMisc* ms, float* infoc,
                                              const float* ys, size_t gs, size_t bs) {
  const int lane = threadIdx.x & 31;
  // the spans' metadata comes straight from global memory (issued before the
  // logits, so its latency overlaps them)
  int body[2], rank[2], size[2];
  long long off[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int kk = lane + 32 * half;
    const bool valid = kk < d.n;
    body[half] = valid ? __ldg(P.body_len + bs + d.a + kk) : 0;
    rank[half] = valid ? __ldg(P.rec_rank + gs + d.a + kk) : 0;
    off[half] = valid ? __ldg(P.rec_off + gs + d.a + kk) : 0;
  }
  const unsigned long long hits = route_hits(page, ys, ms->theta, P.G);
  // expanded spans of this page: entries compacted at [d.a, d.a + count), in
  // span order, each with the record bytes of the ones before it (cum)
  bool ex[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int kk = lane + 32 * half;
    const bool valid = kk < d.n;
    ex[half] = valid && body[half] > 0 && ((hits >> kk) & 1ull);
    if (valid) infoc[d.a - k0 + kk] = (body[half] > 0 && !ex[half]) ? log2f(float(body[half])) : kNegInf;
    size[half] = ex[half] ? int(record_bytes(body[half], rank[half] & 0xffff, (rank[half] >> 16) & 0xffff)) : 0;
  }
  const uint32_t b0 = __ballot_sync(0xffffffffu, ex[0]), b1 = __ballot_sync(0xffffffffu, ex[1]);
  const uint32_t lt = (1u << lane) - 1u;
  // record bytes of one page stay far below 2^31: 32-bit scans
  int incl0 = size[0], incl1 = size[1];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v0 = __shfl_up_sync(0xffffffffu, incl0, o);
    const int v1 = __shfl_up_sync(0xffffffffu, incl1, o);
    if (lane >= o) {
      incl0 += v0;
      incl1 += v1;
    }
  }
  const int tot0 = __shfl_sync(0xffffffffu, incl0, 31);
  const int tot1 = __shfl_sync(0xffffffffu, incl1, 31);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (ex[half]) {
      const int idx = half ? __popc(b0) + __popc(b1 & lt) : __popc(b0 & lt);
      const int cum = half ? tot0 + incl1 - size[1] : incl0 - size[0];
      int4* dst = reinterpret_cast<int4*>(P.entries + gs + d.a + idx);
      dst[0] = make_int4(d.a + lane + 32 * half, body[half], rank[half], 0);
      dst[1] = make_int4(int(uint32_t(off[half])), int(off[half] >> 32), cum, 0);
    }
  }
  const unsigned long long mask = (unsigned long long)b0 | ((unsigned long long)b1 << 32);
  const long long bytes = (long long)tot0 + tot1;
  if (lane == 0) {
    ms->rmask[d.flag] = mask;
    ms->rbytes[d.flag] = bytes;
  }
}

// After every warp has passed its routing pages: publish this CTA's
// expansion summary (per-page masks and bytes, totals) for the producers of
// all CTAs of this KV head.  Warp 0 only.
__device__ __forceinline__ void publish_routes(const DecodeParams& P, SmemMisc* ms, int g, int j,
                                               int np) {
  const int lane = threadIdx.x & 31;
  int cnt = 0;
  long long bytes = 0;
  const size_t pb = (size_t(g) * P.cg + j) * kMaxRoutePages;
  for (int p = lane; p < np; p += 32) {
    const unsigned long long m = ms->rmask[p];
    P.pmask[pb + p] = m;
    P.pbytes[pb + p] = ms->rbytes[p];
    cnt += __popcll(m);
    bytes += ms->rbytes[p];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
  }
  if (lane == 0) {
    P.cta_n[size_t(g) * P.cg + j] = cnt;
    P.cta_bytes[size_t(g) * P.cg + j] = bytes;
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) atomicAdd(&P.groups[g].published, 1);
}

template <int KS>
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
  float* ys = reinterpret_cast<float*>(smem + kOffScratch + 4096);  // routing pages

  if (P.fused) {
    // Run the routing routine once on whatever the W_r area holds (the
    // result is discarded): its code is fetched into the instruction cache
    // while the routing weights and the first routing pages are in flight.
    const unsigned long long warm = route_hits(smem + kOffWr, ys, ms->theta, G);
    if (lane == 0) ms->warm[w] = uint32_t(warm);
  }
  pdl_wait();
  WarpAcc A;
  const __nv_bfloat16* qg = P.q + (size_t(b) * P.Hq + size_t(c) * G) * kHeadDim;
  // query A fragments of this lane (rows 0..7 = heads, zero past G), grouped
  // by 32 head dims; stored to the warp's scratch once the prologue is done
  uint4 qf[4];
  {
    const int r0 = lane >> 2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = 32 * i + 2 * (lane & 3);
      const __nv_bfloat16* qr = qg + r0 * kHeadDim + k;
      qf[i].x = r0 < G ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
      qf[i].y = r0 < G ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
      qf[i].z = r0 < G ? *reinterpret_cast<const uint32_t*>(qr + 16) : 0u;
      qf[i].w = r0 < G ? *reinterpret_cast<const uint32_t*>(qr + 24) : 0u;
    }
  }
#pragma unroll
  for (int t = 0; t < 16; ++t) A.o[t][0] = A.o[t][1] = 0.f;
  A.m_row = kNegInf;
  A.l_part = 0.f;
  ExpAcc<KS> X;
  X.had = false;

  if (P.fused) {
    if (tid < 8) ms->theta[tid] = tid < G ? P.theta[c * G + tid] : 0.f;
    if (!mbar_wait(&ms->wr_bar, 0, kWaitLimit) && tid == 0)
      set_device_error(P.status, DEV_WAIT_TIMEOUT, 5);
    // y_h = W_r[c] q_h on the tensor cores: heads are the M rows, warp w takes
    // routing coordinates 16w .. 16w+15 (two n-tiles); W_r (fp32, in four
    // 128B-swizzled boxes of 64 rows x 32 floats) is split into bf16 hi + lo
    const int gid = lane >> 2, tig = lane & 3;
    float yh[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, yl[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t a0 = (ks & 1) ? qf[ks >> 1].z : qf[ks >> 1].x;
      const uint32_t a2 = (ks & 1) ? qf[ks >> 1].w : qf[ks >> 1].y;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int r = 16 * w + 8 * nt + gid;
        uint32_t bh[2], bl[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int d = 16 * ks + 8 * hf + 2 * tig;
          const float2 v = *reinterpret_cast<const float2*>(
              smem + kOffWr + (d >> 5) * 8192 + r * 128 + ((((d & 31) >> 2) ^ (r & 7)) << 4) +
              (d & 3) * 4);
          split_bf16(v.x, v.y, bh[hf], bl[hf]);
        }
        mma_bf16_rows8(yh[nt][0], yh[nt][1], a0, a2, bh[0], bh[1]);
        mma_bf16_rows8(yl[nt][0], yl[nt][1], a0, a2, bl[0], bl[1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int r = 16 * w + 8 * nt + 2 * tig;
      ys[gid * kRouteDim + r] = yh[nt][0] + yl[nt][0];
      ys[gid * kRouteDim + r + 1] = yh[nt][1] + yl[nt][1];
    }
    named_bar(1, kConsumers);
  }

  // the routing weights are consumed: their space becomes per-warp scratch
  A.qfrag = smem_u32(smem + kOffWr + w * 8192);
#pragma unroll
  for (int i = 0; i < 4; ++i) sts128(A.qfrag + (i * 32 + lane) * 16, qf[i]);
  __syncwarp();

  // this warp's ring: slots 2w, 2w+1
  Ring R;
  bool routed = false;  // passed the routing barrier
  const int np = (k1 - k0 + kRouteSpans - 1) / kRouteSpans;
  for (;;) {
    const int slot = w * kSlotsPerWarp + R.s;
    if (!mbar_wait_parked(&ms->full[slot], R.phase)) {
      if (lane == 0) set_device_error(P.status, DEV_WAIT_TIMEOUT, 4);
      if (!routed) named_bar(2, kConsumers);
      break;
    }
    const PageDesc d = ms->desc[slot];
    const uint8_t* page = slot_ptr(smem, slot);
    const uint32_t pu = smem_u32(page);
    if (!routed && (d.type == PG_SYNC || d.type == PG_END)) {
      // all routing pages of the CTA are done past this barrier; warp 0's
      // gpu-scope fence after it (in publish_routes) is cumulative, so it
      // also orders the other warps' entry writes before the publication
      named_bar(2, kConsumers);
      routed = true;
      if (P.fused && w == 0 && d.type == PG_SYNC) publish_routes(P, ms, g, j, np);
    }
    // one call site per page routine keeps the kernel's code small
    if (d.type == PG_ROUTE) {
      consume_route(page, d, k0, P, ms, infoc, ys, gs, size_t(b) * P.max_spans);
    } else if (d.type == PG_INFO) {
      const uint16_t* src = reinterpret_cast<const uint16_t*>(page);
      for (int i = lane; i < d.n; i += 32) {
        const int inf = src[i], body = inf & 0x7fff;
        infoc[i] = (body > 0 && !(inf & 0x8000)) ? log2f(float(body)) : kNegInf;
      }
    } else if (d.type == PG_FULL || d.type == PG_SUM) {
      consume_kv_page(A, pu, pu + 2 * kBoxBytes, d.n,
                      d.type == PG_SUM ? infoc + (d.a - k0) : nullptr, P.scale_log2);
    } else if (d.type == PG_EXP || d.type == PG_EXPM) {
      // PG_EXP: one part of a record split over pages; PG_EXPM: whole records.
      // The next part of a split record goes into this warp's other slot
      // (its previous page is consumed) before this part is processed.
      if (d.type == PG_EXP && lane == 0 && d.part + 1 < split_nparts(d.b, d.rk, d.rv))
        issue_split_part(smem, ms, P, w * kSlotsPerWarp + (R.s ^ 1), d.part + 1, d.b, d.rk, d.rv,
                         d.src);
      const int nrec = d.type == PG_EXPM ? d.n : 1;
      for (int i = 0; i < nrec; ++i) {
        int off_a = d.off_a, off_uk = d.off_uk, off_uv = d.off_uv, off_b = d.off_b;
        int n = d.n, rk = d.rk, rv = d.rv;
        if (d.type == PG_EXPM) {
          const RecInfo ri = ms->rec[slot][i];
          const RecordLayout RL = record_layout(ri.b, ri.rk, ri.rv);
          off_a = ri.off;
          off_uk = ri.off + int(RL.uk);
          off_uv = ri.off + int(RL.uv);
          off_b = ri.off + int(RL.vpart);
          n = ri.b;
          rk = ri.rk;
          rv = ri.rv;
        }
        if (off_a >= 0) exp_key<KS>(A, X, page + off_a, rk, P.scale_log2);
        if (n > 0) exp_tokens<KS>(A, X, page + off_uk, page + off_uv, n, rk, rv);
        if (off_b >= 0) exp_value<KS>(A, X, page + off_b, rv);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->empty[slot]);
    // the last part of a split record consumed: the ring is the producer's again
    if (d.type == PG_EXP && lane == 0 && d.part + 1 == split_nparts(d.b, d.rk, d.rv))
      st_release_cta(&ms->sp_busy[w], 0);
    if (d.type == PG_END) break;
    ring_advance(R);
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
  // (the partials arrive by bulk copy, chunks of kCombineChunk CTAs, so the
  // merge costs one global round trip per chunk)
  __threadfence();
  const int cg = P.cg;
  const Partial* parts = P.partials + size_t(g) * cg;
  float* sm_s = reinterpret_cast<float*>(smem + kOffInfo);          // [cg][8] m, then scales
  float* sm_l = reinterpret_cast<float*>(smem + kCombineLOff);      // [cg][8]
  float* sm_ML = reinterpret_cast<float*>(smem + kOffScratch);      // M[8], L[8]
  const Partial* cbuf = reinterpret_cast<const Partial*>(smem);     // chunk of partials
  for (int i = tid; i < cg * 8; i += kConsumers) {
    const int jj = i >> 3, h = i & 7;
    sm_s[i] = h < G ? __ldcg(&parts[jj].m[h]) : kNegInf;
    sm_l[i] = h < G ? __ldcg(&parts[jj].l[h]) : 0.f;
  }
  named_bar(1, kConsumers);
  if (tid < G) {
    float M = kNegInf;
    for (int jj = 0; jj < cg; ++jj) M = fmaxf(M, sm_s[jj * 8 + tid]);
    float L = 0.f;
    if (M != kNegInf)
      for (int jj = 0; jj < cg; ++jj) L = fmaf(sm_l[jj * 8 + tid], exp2f(sm_s[jj * 8 + tid] - M), L);
    sm_ML[tid] = M;
    sm_ML[8 + tid] = L;
  }
  named_bar(1, kConsumers);
  for (int i = tid; i < cg * 8; i += kConsumers) {
    const int h = i & 7;
    const float M = h < G ? sm_ML[h] : kNegInf;
    sm_s[i] = (M == kNegInf) ? 0.f : exp2f(sm_s[i] - M);
  }
  float Oh[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) Oh[h] = 0.f;
  for (int c0 = 0, ph = 0; c0 < cg; c0 += kCombineChunk, ph ^= 1) {
    const int nc = (cg - c0) < kCombineChunk ? (cg - c0) : kCombineChunk;
    named_bar(1, kConsumers);  // the previous chunk is consumed, the scales are written
    if (tid == 0) {
      fence_proxy_async_global();
      mbar_arrive_expect_tx(&ms->cmb_bar, uint32_t(nc * sizeof(Partial)));
      bulk_g2s(smem, parts + c0, uint32_t(nc * sizeof(Partial)), &ms->cmb_bar);
    }
    // every thread takes every barrier of this loop, even after a timeout
    const bool landed = mbar_wait(&ms->cmb_bar, uint32_t(ph), kWaitLimit);
    if (!landed && tid == 0) set_device_error(P.status, DEV_WAIT_TIMEOUT, 7);
    for (int jj = 0; landed && jj < nc; ++jj) {
#pragma unroll
      for (int h = 0; h < 8; ++h)
        if (h < G) Oh[h] = fmaf(cbuf[jj].o[h][tid], sm_s[(c0 + jj) * 8 + h], Oh[h]);
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < G) {
      const float L = sm_ML[8 + h];
      const size_t row = size_t(b) * P.Hq + size_t(c) * G + h;
      P.out[row * kHeadDim + tid] = L > 0.f ? Oh[h] / L : 0.f;
      if (tid == 0 && P.lse != nullptr)
        P.lse[row] = L > 0.f ? (sm_ML[h] + log2f(L)) * kLn2 : kNegInf;
    }
  }
  named_bar(1, kConsumers);
  if (P.expanded_out != nullptr && P.fused) {
    // the CTAs' routing pages in order; page p of CTA jj covers spans
    // sk0 + 64p + (0..63), bit i of its mask marks span sk0 + 64p + i
    int* pre = reinterpret_cast<int*>(sm_ML + 16);  // [kMaxRoutePages + 1] (scratch: 6 KB)
    int base = 0;
    for (int jj = 0; jj < cg; ++jj) {
      int a0, a1, sk0, sk1;
      fixed_range(jj, cg, n_full, n_sp, 1, a0, a1, sk0, sk1);
      const int npj = (sk1 - sk0 + kRouteSpans - 1) / kRouteSpans;
      const uint64_t* pm = P.pmask + (size_t(g) * cg + jj) * kMaxRoutePages;
      if (tid == 0) {
        int acc = 0;
        for (int p = 0; p < npj; ++p) {
          pre[p] = acc;
          acc += __popcll(__ldcg(reinterpret_cast<const unsigned long long*>(pm) + p));
        }
        pre[npj] = acc;
      }
      named_bar(1, kConsumers);
      for (int t = tid; t < npj * 64; t += kConsumers) {
        const int p = t >> 6, i = t & 63;
        const unsigned long long m = __ldcg(reinterpret_cast<const unsigned long long*>(pm) + p);
        if ((m >> i) & 1ull)
          P.expanded_out[gs + base + pre[p] + __popcll(m & ((1ull << i) - 1ull))] = sk0 + 64 * p + i;
      }
      base += pre[npj];
      named_bar(1, kConsumers);
    }
    if (tid == 0 && P.n_expanded_out != nullptr) P.n_expanded_out[g] = base;
  }
  named_bar(1, kConsumers);
  if (tid == 0) {
    P.groups[g].published = 0;
    P.groups[g].done = 0;
  }
}

// grid: (cg, Hkv, B); block: 4 consumer warps + 1 producer warp
template <int KS>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  SmemMisc* ms = reinterpret_cast<SmemMisc*>(smem + kOffMisc);
  const int j = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int g = b * P.Hkv + c;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&ms->full[s], 1);
      mbar_init(&ms->empty[s], 1);  // each slot belongs to one consumer warp
    }
    mbar_init(&ms->wr_bar, 1);
    mbar_init(&ms->cmb_bar, 1);
    ms->is_last = 0;
    for (int x = 0; x < kConsumerWarps; ++x) ms->sp_busy[x] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (threadIdx.x >= kConsumers)
    producer_warp(smem, ms, P, g, j, b, c);
  else
    consumer_warps<KS>(smem, ms, P, g, j, b, c);
}

}  // namespace sekv
