// Decode-time maintenance of one layer's span cache (sekv_maint_init,
// sekv_append_token).
//
// SeKV, technical summary (gist.science, German page / Chinese page), and the
// lay explainer of the same pages: the GPU keeps the very last part of the
// text at full resolution (explainer, part 2 / 两层记忆); high-surprisal
// tokens are span boundaries and a span is the run of tokens between two
// neighbouring anchors (Methodik 1 / 方法论 1); each span is kept as a routing
// summary and a gated SVD basis (Methodik 2 / 方法论 2).  During decode the
// new token joins the recent window, the token leaving the window continues
// the segmentation walk, and a span can be built once the next anchor closes
// it.  Closed spans wait, with the open span -- anchor and body -- at full
// resolution in the tail of the full rows, in front of the recent window,
// until a flush builds them all (the caller picks how often).
//
// Row layout of one group (sequence b, KV head c), capacity `cap` rows:
//   [0, n_sink)                 sinks
//   [n_sink, n_sink + n_spans)  anchors of the built spans
//   [n_sink + n_spans, + n_tail) the tail: the closed spans waiting to be
//                               built (anchor and body each), the open span,
//                               then the recent window (oldest first)
// A flush builds the waiting spans as ordinals n_spans, n_spans + 1, ...: each
// keeps its anchor row (moved to row n_sink + k), its body rows leave the
// tail, and the rest of the tail moves up over them.
#include "build.cuh"

namespace sekv {

namespace {

constexpr int kRowChunks = kHeadDim * 2 / 16;  // 16-byte chunks per row

__device__ __forceinline__ int gate_rank_m(const float* g, int R) {
  int r = 0;
  while (r < R && g[r] > 0.5f) ++r;
  return r;
}

// Move rows [from, from + n) of one group's K and V rows to [to, to + n),
// to < from (overlap allowed): chunks of rows in increasing order, each read
// whole into registers before any of it is written, so a chunk never
// overwrites rows a later chunk still has to read.
__device__ void move_rows_down(__nv_bfloat16* Kg, __nv_bfloat16* Vg, int from, int to, int n) {
  constexpr int kPer = 4;  // 16-byte chunks per thread and array per step
  const int step = blockDim.x * kPer;  // chunks per step
  int4* K4 = reinterpret_cast<int4*>(Kg);
  int4* V4 = reinterpret_cast<int4*>(Vg);
  const int total = n * kRowChunks;
  for (int c0 = 0; c0 < total; c0 += step) {
    int4 kv[kPer], vv[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = c0 + threadIdx.x + i * blockDim.x;
      if (e < total) {
        kv[i] = K4[size_t(from) * kRowChunks + e];
        vv[i] = V4[size_t(from) * kRowChunks + e];
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = c0 + threadIdx.x + i * blockDim.x;
      if (e < total) {
        K4[size_t(to) * kRowChunks + e] = kv[i];
        V4[size_t(to) * kRowChunks + e] = vv[i];
      }
    }
    __syncthreads();
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// init, from a prefill build of a prefix of length T: the build closed its
// last span at the end of the middle region; that span is open again (its
// anchor and body return to full resolution from K, V).  grid (Hkv, B).
// pend[b] = {n_spans after, n_tail, s_open}.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) maint_init_rows_kernel(const MaintParams M,
                                                              const __nv_bfloat16* K,
                                                              const __nv_bfloat16* V,
                                                              const float* H) {
  __shared__ int red[8];
  const int c = blockIdx.x, b = blockIdx.y, g = b * M.Hkv + c, tid = threadIdx.x;
  const int n_sp = M.n_spans[b];
  int s = -1;  // the open anchor
  if (n_sp > 0) {
    int acc = 0;
    for (int k = tid; k < n_sp - 1; k += blockDim.x) acc += M.body_len[size_t(b) * M.max_spans + k] + 1;
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((tid & 31) == 0) red[tid >> 5] = acc;
    __syncthreads();
    acc = 0;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) acc += red[w];
    s = M.n_sink + acc;
  }
  const int n_closed = n_sp > 0 ? n_sp - 1 : 0;
  const int start = M.n_sink + n_closed;
  const int src0 = s >= 0 ? s : M.T - M.n_recent;  // first token of the tail
  const int n_tail = M.T - src0;
  if (start + n_tail > M.cap) {
    if (tid == 0) set_device_error(M.status, DEV_STAGING_FULL, b);
    return;
  }
  const int4* Ks = reinterpret_cast<const int4*>(K + (size_t(g) * M.T + src0) * kHeadDim);
  const int4* Vs = reinterpret_cast<const int4*>(V + (size_t(g) * M.T + src0) * kHeadDim);
  int4* Kd = reinterpret_cast<int4*>(M.k_full + (size_t(g) * M.cap + start) * kHeadDim);
  int4* Vd = reinterpret_cast<int4*>(M.v_full + (size_t(g) * M.cap + start) * kHeadDim);
  for (int e = tid; e < n_tail * kRowChunks; e += blockDim.x) {
    Kd[e] = Ks[e];
    Vd[e] = Vs[e];
  }
  if (c == 0) {
    for (int i = tid; i < n_tail; i += blockDim.x)
      M.tail_h[size_t(b) * M.cap + start + i] = H[size_t(b) * M.T + src0 + i];
    if (tid == 0) {
      int32_t* pd = M.pend + size_t(b) * 8;
      pd[0] = n_closed;
      pd[1] = n_tail;
      pd[2] = s;
    }
  }
}

// grid (B): the per-sequence counters, once every group's rows are in place.
__global__ void maint_init_commit_kernel(const MaintParams M) {
  const int b = blockIdx.x;
  if (threadIdx.x != 0) return;
  const int32_t* pd = M.pend + size_t(b) * 8;
  M.n_spans[b] = pd[0];
  M.n_tail[b] = pd[1];
  M.s_open[b] = pd[2];
  M.seq_len[b] = M.T;
}

// grid (B*Hkv): the end of the records in the store (their maximum end).
__global__ void __launch_bounds__(256) maint_used_kernel(const MaintParams M) {
  const int g = blockIdx.x, b = g / M.Hkv;
  const int n_sp = M.n_spans[b];
  unsigned long long mx = 0;
  for (int k = threadIdx.x; k < n_sp; k += blockDim.x) {
    const size_t gk = size_t(g) * M.max_spans + k;
    const int bl = M.body_len[size_t(b) * M.max_spans + k];
    const int rk = M.rec_rank[gk] & 0xffff, rv = (M.rec_rank[gk] >> 16) & 0xffff;
    if (bl > 0) {
      const unsigned long long e = (unsigned long long)M.rec_off[gk] + record_bytes(bl, rk, rv);
      mx = e > mx ? e : mx;
    }
  }
  if (mx) atomicMax(M.store_used, mx);
}

// ---------------------------------------------------------------------------
// one append (grid (B), one CTA per sequence, so that the sequence's counters
// have a single reader and writer): the new token's rows at the end of the
// tail; the segmentation decision for the token leaving the recent window
// (t = T - n_recent, T the length before the append); a span this closes
// joins the waiting spans.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) maint_append_kernel(const MaintParams M) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int n_sp = M.n_spans[b], n_tail = M.n_tail[b], s = M.s_open[b], T = M.seq_len[b];
  const int np = M.n_pend[b], prow = M.pend_rows[b];
  const int row0 = M.n_sink + n_sp;  // the tail's first row
  const int r_new = row0 + n_tail;
  if (r_new >= M.cap) {
    if (tid == 0) set_device_error(M.status, DEV_STAGING_FULL, b);
    return;
  }
  // the new token's key and value, every KV head
  for (int e = tid; e < M.Hkv * 2 * 16; e += blockDim.x) {
    const int c = e / 32, half = (e / 16) & 1, q = e & 15;
    const size_t g = size_t(b) * M.Hkv + c;
    const int4* src = reinterpret_cast<const int4*>((half ? M.v_new : M.k_new) + g * kHeadDim);
    int4* dst = reinterpret_cast<int4*>((half ? M.v_full : M.k_full) +
                                        (g * M.cap + r_new) * kHeadDim);
    dst[q] = src[q];
  }
  if (tid != 0) return;
  M.tail_h[size_t(b) * M.cap + r_new] = M.h_new[b];
  const int t = T - M.n_recent;
  if (t >= M.n_sink) {
    if (s < 0) {
      M.s_open[b] = t;  // the first middle token opens span 0
    } else {
      const int n = t - s;
      const float h = M.tail_h[size_t(b) * M.cap + row0 + prow + n];  // token t's row
      if ((h > M.tau && n >= M.len_min) || n == M.len_max) {
        if (np >= kMaxPending || n_sp + np + 1 > M.max_spans) {
          set_device_error(M.status, DEV_STAGING_FULL, b);  // flush first
        } else {
          M.pend_len[size_t(b) * kMaxPending + np] = n;
          M.n_pend[b] = np + 1;
          M.pend_rows[b] = prow + n;
          M.s_open[b] = t;
        }
      }
    }
  }
  M.n_tail[b] = n_tail + 1;
  M.seq_len[b] = T + 1;
}

// ---------------------------------------------------------------------------
// flush, step 1 (grid (Hkv, B)): per waiting span j of the sequence, ordinal
// k = n_spans + j, anchor row n_sink + n_spans + (rows of the spans before
// it): its ranks from the gates, its record's place at the end of the store,
// its SVD work items; the sequence's span arrays (anchor row, body) and the
// range the summaries cover.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMaxPending) maint_flush_plan_kernel(const MaintParams M) {
  __shared__ int pre[kMaxPending];
  const int c = blockIdx.x, b = blockIdx.y, g = b * M.Hkv + c, j = threadIdx.x;
  const int n_sp = M.n_spans[b], np = M.n_pend[b];
  const int len = j < np ? M.pend_len[size_t(b) * kMaxPending + j] : 0;
  pre[j] = len;
  __syncthreads();
  for (int o = 1; o < kMaxPending; o <<= 1) {  // inclusive scan of the lengths
    const int v = j >= o ? pre[j - o] : 0;
    __syncthreads();
    pre[j] += v;
    __syncthreads();
  }
  if (j == 0) M.gbase[g] = 0;
  if (c == 0 && j == 0) {
    M.only_k[b] = n_sp;
    M.only_n[b] = np;
  }
  if (j >= np) return;
  const int k = n_sp + j, bl = len - 1;
  const int anchor_row = M.n_sink + n_sp + (pre[j] - len);
  const size_t gk = size_t(g) * M.max_spans + k;
  int rk = 0, rv = 0;
  if (bl > 0) {
    const int R = bl < M.rank_cap ? bl : M.rank_cap;
    const float* gkp = M.gates + ((size_t(b) * M.Hkv + c) * 2 * M.max_spans + k) * M.rank_cap;
    rk = gate_rank_m(gkp, R);
    rv = gate_rank_m(gkp + size_t(M.max_spans) * M.rank_cap, R);
    const long long size = record_bytes(bl, rk, rv);
    const unsigned long long off = atomicAdd(M.store_used, (unsigned long long)size);
    if ((long long)off + size > M.store_capacity)
      set_device_error(M.status, DEV_STAGING_FULL, int((off + size) >> 20));
    M.rel_off[gk] = (long long)off;
    const int cls = bl <= 32 ? 0 : bl <= 64 ? 1 : bl <= 128 ? 2 : 3;
    const int pos = atomicAdd(&M.counters[cls], 2);
    if (pos + 1 < M.cls_cap) {
      int32_t* lst = M.cls_list + size_t(cls) * M.cls_cap;
      lst[pos] = int32_t(gk * 2);
      lst[pos + 1] = int32_t(gk * 2 + 1);
    }
  }
  M.rec_rank[gk] = rk | (rv << 16);
  if (c == 0) {
    M.starts[size_t(b) * M.max_spans + k] = anchor_row;
    M.body_len[size_t(b) * M.max_spans + k] = bl;
  }
}

// ---------------------------------------------------------------------------
// flush, last step but one (grid (Hkv, B)), after the summaries and bases are
// built: the waiting spans' anchor rows move to rows n_sink + n_spans + j, in
// increasing j (a destination never lies above its source, nor on a later
// anchor), then the rest of the tail (open span and recent window) moves up
// behind them; the surprisal by row moves along (KV head 0).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) maint_flush_move_kernel(const MaintParams M) {
  const int c = blockIdx.x, b = blockIdx.y, g = b * M.Hkv + c, tid = threadIdx.x;
  const int n_sp = M.n_spans[b], np = M.n_pend[b], prow = M.pend_rows[b];
  const int n_tail = M.n_tail[b];
  if (np == 0) return;
  const int row0 = M.n_sink + n_sp;
  __nv_bfloat16* Kg = M.k_full + size_t(g) * M.cap * kHeadDim;
  __nv_bfloat16* Vg = M.v_full + size_t(g) * M.cap * kHeadDim;
  float* th = M.tail_h + size_t(b) * M.cap;
  int4* K4 = reinterpret_cast<int4*>(Kg);
  int4* V4 = reinterpret_cast<int4*>(Vg);
  // anchors, 8 per step (16 threads per row and array), read before written
  int src = row0;  // anchor row of span j (row0 + the rows of the spans before j)
  for (int j0 = 0; j0 < np; j0 += 8) {
    // the source rows of anchors j0 .. j0 + 7: each thread finds its own
    const int j = j0 + (tid >> 5), q = tid & 15, half = (tid >> 4) & 1;
    int my_src = src;
    for (int i = j0; i < j && i < np; ++i) my_src += M.pend_len[size_t(b) * kMaxPending + i];
    int4 v = make_int4(0, 0, 0, 0);
    float hv = 0.f;
    if (j < np) {
      v = (half ? V4 : K4)[size_t(my_src) * kRowChunks + q];
      hv = th[my_src];
    }
    __syncthreads();
    if (j < np) {
      (half ? V4 : K4)[size_t(row0 + j) * kRowChunks + q] = v;
      if (c == 0 && q == 0 && half == 0) th[row0 + j] = hv;
    }
    __syncthreads();
    for (int i = j0; i < j0 + 8 && i < np; ++i) src += M.pend_len[size_t(b) * kMaxPending + i];
  }
  // the rest of the tail: rows [row0 + prow, row0 + n_tail) -> [row0 + np, ...)
  const int cnt = n_tail - prow;
  if (cnt > 0 && prow > np) {
    move_rows_down(Kg, Vg, row0 + prow, row0 + np, cnt);
    if (c == 0) {
      float hv4[4];
      for (int i0 = 0; i0 < cnt; i0 += 4 * blockDim.x) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int i = i0 + tid + jj * blockDim.x;
          hv4[jj] = i < cnt ? th[row0 + prow + i] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int i = i0 + tid + jj * blockDim.x;
          if (i < cnt) th[row0 + np + i] = hv4[jj];
        }
        __syncthreads();
      }
    }
  }
}

// flush, last step (grid (B)): the sequence's counters.
__global__ void maint_flush_commit_kernel(const MaintParams M) {
  const int b = blockIdx.x;
  if (threadIdx.x != 0) return;
  const int np = M.n_pend[b];
  if (np == 0) return;
  M.n_spans[b] += np;
  M.n_tail[b] -= M.pend_rows[b];  // anchors and bodies: the anchors now count as spans
  M.n_pend[b] = 0;
  M.pend_rows[b] = 0;
}

}  // namespace sekv
