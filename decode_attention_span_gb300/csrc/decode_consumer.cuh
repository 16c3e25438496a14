// Consumer warps of the decode kernel: routing and the online softmax.
//
// The routines are written rolled (runtime loops, one copy of each body):
// the whole kernel's code has to stay resident in the SM's instruction cache
// while four warps run different routines at once.  Operands a rolled loop
// indexes (the query fragments) sit in a small per-warp shared scratch.
#pragma once

#include "decode_attn.cuh"

namespace sekv {

constexpr float kNegInf = -__builtin_huge_valf();

struct WarpAcc {
  float o[16][2];  // output accumulator, row r0 = lane/4, dims 8t + 2(lane%4) + {0,1}
  float m_row;     // running max of row r0 (log2 domain)
  float l_part;    // this lane's share of the row sum
  uint32_t qfrag;  // shared address of this warp's query A fragments (4 x 32 lanes x 16 B)
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

// exp2 of (x - m) that treats an all -inf row as contributing nothing.
__device__ __forceinline__ void softmax_rescale(float m_old, float m_new, float& alpha,
                                                float& msub) {
  if (m_new == kNegInf) {
    alpha = 1.f;
    msub = 0.f;
  } else {
    alpha = exp2f(m_old - m_new);
    msub = m_new;
  }
}

__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16(x0 - hf.x, x1 - hf.y);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Lazy online-softmax re-basing: the running max m only moves when a new
// logit exceeds it by more than kRebase (log2 units), so exponentials stay
// below 2^kRebase and most tiles skip the shuffles and the rescale.  The
// output is normalised by the sum taken against the same m, so the choice of
// m changes only rounding.
constexpr float kRebase = 8.f;

// Re-base the warp's state to cover the row maxima mx (rows lane/4) if
// some lane's exceeds the running max by more than kRebase; returns alpha
// (1 when nothing moved).
__device__ __forceinline__ float rebase_if_needed(WarpAcc& A, float mx) {
  float alpha = 1.f;
  if (__any_sync(0xffffffffu, mx > A.m_row + kRebase)) {
    mx = quad_max(mx);
    const float m_new = fmaxf(A.m_row, mx);
    float msub;
    softmax_rescale(A.m_row, m_new, alpha, msub);
    A.m_row = m_new;
    A.l_part *= alpha;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      A.o[t][0] *= alpha;
      A.o[t][1] *= alpha;
    }
  }
  return alpha;
}

// One tile of 16 full-resolution or summary rows whose two 128-byte halves
// sit in 128B-swizzled boxes `half` bytes apart (keys: dims 0-63 at kb,
// 64-127 at kb + half; values likewise at vb; kb and vb point at the tile's
// first row, and a box's swizzle runs on in its later rows), folded into the
// warp's softmax state with at most one rescale.  bias_row: for summary pages
// the logit bias of the page's spans (log2|S|, or -inf for a span that does
// not enter as a summary); nullptr for full rows.  Rows >= n are masked.
__device__ __forceinline__ void consume_rows16(WarpAcc& A, uint32_t kb, uint32_t vb, int n,
                                               const float* bias_row, float scale_log2,
                                               int half) {
  const int lane = threadIdx.x & 31;
  float s[2][2];
  s[0][0] = s[0][1] = s[1][0] = s[1][1] = 0.f;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {  // 32 head dims per step
    const uint4 q = lds128(A.qfrag + (i * 32 + lane) * 16);
    const uint32_t box = kb + (i >> 1) * half;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(swz128(box, 8 * nt + (lane & 7), (i & 1) * 4 + (lane >> 3)), b0, b1, b2, b3);
      mma_bf16_rows8(s[nt][0], s[nt][1], q.x, q.y, b0, b1);
      mma_bf16_rows8(s[nt][0], s[nt][1], q.z, q.w, b2, b3);
    }
  }
  float mx = kNegInf;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = 8 * nt + 2 * (lane & 3) + e;
      bool valid = key < n;
      float bias = 0.f;
      if (bias_row != nullptr && valid) {
        bias = bias_row[key];
        valid = bias != kNegInf;
      }
      s[nt][e] = valid ? fmaf(s[nt][e], scale_log2, bias) : kNegInf;
      mx = fmaxf(mx, s[nt][e]);
    }
  rebase_if_needed(A, mx);
  const float msub = A.m_row == kNegInf ? 0.f : A.m_row;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) s[nt][e] = ex2_approx(s[nt][e] - msub);
  A.l_part += (s[0][0] + s[0][1]) + (s[1][0] + s[1][1]);
  const int mi = lane >> 3;
  const uint32_t a0 = pack_bf16(s[0][0], s[0][1]);
  const uint32_t a2 = pack_bf16(s[1][0], s[1][1]);
  // value rows past n (zero fill or unrelated rows) must not reach o
  const int kt = 2 * (lane & 3);
  const uint32_t t0 = (kt < n ? 0xffffu : 0u) | (kt + 1 < n ? 0xffff0000u : 0u);
  const uint32_t t1 = (kt + 8 < n ? 0xffffu : 0u) | (kt + 9 < n ? 0xffff0000u : 0u);
  const int key = 8 * (mi & 1) + (lane & 7);
#pragma unroll
  for (int dp = 0; dp < 8; ++dp) {
    const int d0 = 16 * dp;
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(swz128(vb + (d0 >> 6) * half, key, ((d0 & 63) >> 3) + (mi >> 1)), b0, b1, b2, b3);
    b0 &= t0; b2 &= t0; b1 &= t1; b3 &= t1;
    mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], a0, a2, b0, b1);
    mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], a0, a2, b2, b3);
  }
}

// Routing logits z[span][head] = s_span . y_head of a routing page (two
// 128B-swizzled boxes of 32 rows x 32 floats: routing dims 0-31, then 32-63)
// in fp32 FMAs, lane l taking span l, four heads per pass (y rows past the
// group are zero and ignored).  Chunk c of a row sits at c ^ (row & 7), so
// eight lanes read eight different bank groups; the y reads are broadcasts.
// Returns whether some head h of the group has z > theta_h for this lane's
// span (rows past the page's spans are computed and ignored by the caller).
__device__ __forceinline__ bool route32(const uint8_t* page, const float* ys, const float* theta,
                                        int G) {
  const int lane = threadIdx.x & 31, sw = lane & 7;
  bool hit = false;
#pragma unroll 1
  for (int h0 = 0; h0 < G; h0 += 4) {
    float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int c = 0; c < 16; ++c) {  // routing dims 4c .. 4c + 3
      const float4 s = *reinterpret_cast<const float4*>(page + (c >> 3) * 4096 + lane * 128 +
                                                        (((c & 7) ^ sw) << 4));
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const float4 y = *reinterpret_cast<const float4*>(ys + (h0 + hh) * kRouteDim + 4 * c);
        z[hh] = fmaf(s.w, y.w, fmaf(s.z, y.z, fmaf(s.y, y.y, fmaf(s.x, y.x, z[hh]))));
      }
    }
#pragma unroll
    for (int hh = 0; hh < 4; ++hh)
      if (h0 + hh < G) hit |= z[hh] > theta[h0 + hh];
  }
  return hit;
}

// ---------------------------------------------------------------------------
// Expanded spans, all on the tensor cores (query heads = M rows):
//   key part:    c = diag(sigma_K g_K) Vt_K q  (scale*log2(e) folded in),
//                kept as bf16 hi + lo A fragments (near-fp32 precision)
//   body tokens: logits = c^T U_K^T, softmax, w += p^T U_V
//   value part:  o += diag(sigma_V g_V) w  times Vt_V (hi + lo)
// One warp handles a whole record.  KS = rank k-steps of 16 (ranks up to
// 16 KS): every loop has a fixed trip count; ranks past the record's own are
// masked arithmetically (no data-dependent branches in the inner loops).
// ---------------------------------------------------------------------------
template <int KS>
struct ExpAcc {
  uint32_t ch[KS][2];    // c hi A-fragments for k-steps of 16 ranks: {a0, a2}
  uint32_t cl[KS][2];    // c lo parts
  float wacc[2 * KS][2];  // w (heads x rV) in C layout: tile jt = columns 8jt..8jt+7
  bool had;
};

// Masks of the bf16 pairs a lane holds in a B fragment of k-step ks whose
// k index is a rank: pair j, j+1 (m0) and j+8, j+9 (m1), j = 16 ks + 2 (lane%4).
__device__ __forceinline__ void rank_masks(int ks, int r, uint32_t& m0, uint32_t& m1) {
  const int j = 16 * ks + 2 * (threadIdx.x & 3);
  m0 = (j < r ? 0xffffu : 0u) | (j + 1 < r ? 0xffff0000u : 0u);
  m1 = (j + 8 < r ? 0xffffu : 0u) | (j + 9 < r ? 0xffff0000u : 0u);
}

template <int KS>
__device__ __forceinline__ void exp_key(const WarpAcc& A, ExpAcc<KS>& X, const uint8_t* part,
                                        int rK, float scale_log2) {
  const int lane = threadIdx.x & 31;
  const float* sig = reinterpret_cast<const float*>(part + 16);
  const float* gat = sig + r4(rK);
  const uint32_t vt = smem_u32(part + 16 + 8 * r4(rK));
  float cv[2 * KS][2];
#pragma unroll
  for (int nt = 0; nt < 2 * KS; ++nt) cv[nt][0] = cv[nt][1] = 0.f;
  uint4 qv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) qv[i] = lds128(A.qfrag + (i * 32 + lane) * 16);
  // Vt_K rows past rK read the record's next bytes; their columns of c are
  // dropped by the selects below
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // 32 head dims per step
#pragma unroll
    for (int nt = 0; nt < 2 * KS; ++nt) {
      uint32_t b0, b1, b2, b3;
      const int row = 8 * nt + (lane & 7), chunk = 4 * i + (lane >> 3);
      ldsm_x4(vt + row * 256 + ((chunk ^ (row & 7)) << 4), b0, b1, b2, b3);
      mma_bf16_rows8(cv[nt][0], cv[nt][1], qv[i].x, qv[i].y, b0, b1);
      mma_bf16_rows8(cv[nt][0], cv[nt][1], qv[i].z, qv[i].w, b2, b3);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2 * KS; ++nt) {
    const int j0 = 8 * nt + 2 * (lane & 3);
    cv[nt][0] = j0 < rK ? cv[nt][0] * sig[j0] * gat[j0] * scale_log2 : 0.f;
    cv[nt][1] = j0 + 1 < rK ? cv[nt][1] * sig[j0 + 1] * gat[j0 + 1] * scale_log2 : 0.f;
  }
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    split_bf16(cv[2 * ks][0], cv[2 * ks][1], X.ch[ks][0], X.cl[ks][0]);
    split_bf16(cv[2 * ks + 1][0], cv[2 * ks + 1][1], X.ch[ks][1], X.cl[ks][1]);
  }
#pragma unroll
  for (int t = 0; t < 2 * KS; ++t) X.wacc[t][0] = X.wacc[t][1] = 0.f;
  X.had = false;
}


// Scores (log2 domain, scale folded into c) of the 16 body tokens
// [rbase, rbase + 16) for the query heads, C layout: s[nt][e] is head
// lane/4, token rbase + 8 nt + 2 (lane%4) + e; tokens >= n get -inf.
template <int KS>
__device__ __forceinline__ void token_scores(const ExpAcc<KS>& X, uint32_t uku, int sk,
                                             int rbase, int n, int rK, float (&s)[2][2]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3;
  s[0][0] = s[0][1] = s[1][0] = s[1][1] = 0.f;
  const int tok = rbase + 8 * (mi >> 1) + (lane & 7);
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t b0, b1, b2, b3, m0, m1;
    ldsm_x4(uku + tok * sk + (2 * ks + (mi & 1)) * 16, b0, b1, b2, b3);
    rank_masks(ks, rK, m0, m1);
    b0 &= m0; b2 &= m0; b1 &= m1; b3 &= m1;
    mma_bf16_rows8(s[0][0], s[0][1], X.ch[ks][0], X.ch[ks][1], b0, b1);
    mma_bf16_rows8(s[1][0], s[1][1], X.ch[ks][0], X.ch[ks][1], b2, b3);
    mma_bf16_rows8(s[0][0], s[0][1], X.cl[ks][0], X.cl[ks][1], b0, b1);
    mma_bf16_rows8(s[1][0], s[1][1], X.cl[ks][0], X.cl[ks][1], b2, b3);
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (rbase + 8 * nt + 2 * (lane & 3) + e >= n) s[nt][e] = kNegInf;
}

// Body tokens [0, n) of this page; U_K rows at uk, U_V rows at uv (row
// strides r8(rK), r8(rV) bf16), one pass of 16-token tiles with lazy
// re-basing (the tiles are independent unless a re-base is needed).  Rows
// or ranks past the valid ones read neighbouring shared memory and are
// masked, never multiplied.
template <int KS>
__device__ __forceinline__ void exp_tokens(WarpAcc& A, ExpAcc<KS>& X, const uint8_t* uk,
                                           const uint8_t* uv, int n, int rK, int rV) {
  if (n <= 0) return;
  const int lane = threadIdx.x & 31;
  const int sk = 2 * r8(rK), sv = 2 * r8(rV);  // row strides in bytes
  const uint32_t uku = smem_u32(uk), uvu = smem_u32(uv);
  const int mi = lane >> 3;
  X.had = true;
#pragma unroll 2
  for (int rb = 0; rb < n; rb += 16) {
    float s[2][2];
    token_scores<KS>(X, uku, sk, rb, n, rK, s);
    const float alpha =
        rebase_if_needed(A, fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1])));
    if (alpha != 1.f) {
#pragma unroll
      for (int t = 0; t < 2 * KS; ++t) {
        X.wacc[t][0] *= alpha;
        X.wacc[t][1] *= alpha;
      }
    }
    const float msub = A.m_row == kNegInf ? 0.f : A.m_row;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) s[nt][e] = ex2_approx(s[nt][e] - msub);
    // into the running sum right away: a later re-base rescales it
    A.l_part += (s[0][0] + s[0][1]) + (s[1][0] + s[1][1]);
    const uint32_t a0 = pack_bf16(s[0][0], s[0][1]);
    const uint32_t a2 = pack_bf16(s[1][0], s[1][1]);
    const int tk = rb + 2 * (lane & 3);  // tokens held by b0/b2 (+8 in b1/b3)
    const uint32_t t0 = (tk < n ? 0xffffu : 0u) | (tk + 1 < n ? 0xffff0000u : 0u);
    const uint32_t t1 = (tk + 8 < n ? 0xffffu : 0u) | (tk + 9 < n ? 0xffff0000u : 0u);
    const int tok = rb + 8 * (mi & 1) + (lane & 7);
#pragma unroll
    for (int jp = 0; jp < KS; ++jp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(uvu + tok * sv + (2 * jp + (mi >> 1)) * 16, b0, b1, b2, b3);
      b0 &= t0; b2 &= t0; b1 &= t1; b3 &= t1;
      mma_bf16_rows8(X.wacc[2 * jp][0], X.wacc[2 * jp][1], a0, a2, b0, b1);
      mma_bf16_rows8(X.wacc[2 * jp + 1][0], X.wacc[2 * jp + 1][1], a0, a2, b2, b3);
    }
  }
}

template <int KS>
__device__ __forceinline__ void exp_value(WarpAcc& A, ExpAcc<KS>& X, const uint8_t* part,
                                          int rV) {
  if (!X.had) return;
  const int lane = threadIdx.x & 31;
  const float* sig = reinterpret_cast<const float*>(part);
  const float* gat = sig + r4(rV);
  const uint32_t vt = smem_u32(part + 8 * r4(rV));
  const int mi = lane >> 3;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    // coefficients of ranks 16 ks .. 16 ks + 15 as A fragments, hi and lo
    const int j0 = 16 * ks + 2 * (lane & 3);
    const float c0 = j0 < rV ? X.wacc[2 * ks][0] * sig[j0] * gat[j0] : 0.f;
    const float c1 = j0 + 1 < rV ? X.wacc[2 * ks][1] * sig[j0 + 1] * gat[j0 + 1] : 0.f;
    const float c2 = j0 + 8 < rV ? X.wacc[2 * ks + 1][0] * sig[j0 + 8] * gat[j0 + 8] : 0.f;
    const float c3 = j0 + 9 < rV ? X.wacc[2 * ks + 1][1] * sig[j0 + 9] * gat[j0 + 9] : 0.f;
    uint32_t h0, l0, h2, l2, m0, m1;
    split_bf16(c0, c1, h0, l0);
    split_bf16(c2, c3, h2, l2);
    rank_masks(ks, rV, m0, m1);
    const int j = 16 * ks + 8 * (mi & 1) + (lane & 7);  // Vt_V row addressed by this lane
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vt + j * 256 + (((2 * dp + (mi >> 1)) ^ (j & 7)) << 4), b0, b1, b2, b3);
      b0 &= m0; b2 &= m0; b1 &= m1; b3 &= m1;
      mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], h0, h2, b0, b1);
      mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], h0, h2, b2, b3);
      mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], l0, l2, b0, b1);
      mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], l0, l2, b2, b3);
    }
  }
}

}  // namespace sekv
