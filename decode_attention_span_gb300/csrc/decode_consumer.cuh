// Consumer warps of the decode kernel: routing and the online softmax.
#pragma once

#include "decode_attn.cuh"

namespace sekv {

constexpr float kNegInf = -__builtin_huge_valf();

struct WarpAcc {
  float o[16][2];   // output accumulator, row r0 = lane/4, dims 8t + 2(lane%4) + {0,1}
  float m_row;      // running max of row r0 (log2 domain)
  float l_part;     // this lane's share of the row sum
  uint32_t qa[8][2];  // query A fragments (rows 0..7), one pair per 16-dim k-step
};

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
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

// One 64-row page of keys (full rows or summaries): warp w takes rows
// 16w..16w+15.  kb: shared address of the key boxes (dims 0-63 at +0, 64-127
// at +8192), vb likewise for values.  bias: for summary pages, the logit bias
// of the page's first span onward (log2|S|, or -inf for a span that does not
// enter as a summary); nullptr for full rows.
__device__ __forceinline__ void consume_kv_tile(WarpAcc& A, uint32_t kb, uint32_t vb, int n,
                                                const float* bias_row, float scale_log2) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int rbase = 16 * w;
  if (rbase >= n) return;
  float s[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, s2[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t box = kb + (i >> 1) * 8192;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(swz128(box, rbase + 8 * nt + (lane & 7), (i & 1) * 4 + (lane >> 3)), b0, b1, b2,
              b3);
      mma_bf16_rows8(s[nt][0], s[nt][1], A.qa[2 * i][0], A.qa[2 * i][1], b0, b1);
      mma_bf16_rows8(s2[nt][0], s2[nt][1], A.qa[2 * i + 1][0], A.qa[2 * i + 1][1], b2, b3);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    s[nt][0] += s2[nt][0];
    s[nt][1] += s2[nt][1];
  }
  float x[2][2];
  float mx = kNegInf;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = rbase + 8 * nt + 2 * (lane & 3) + e;
      bool valid = key < n;
      float bias = 0.f;
      if (bias_row != nullptr && valid) {
        bias = bias_row[key];
        valid = bias != kNegInf;
      }
      x[nt][e] = valid ? fmaf(s[nt][e], scale_log2, bias) : kNegInf;
      mx = fmaxf(mx, x[nt][e]);
    }
  mx = quad_max(mx);
  const float m_new = fmaxf(A.m_row, mx);
  float alpha, msub;
  softmax_rescale(A.m_row, m_new, alpha, msub);
  float p[2][2], ps = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      p[nt][e] = exp2f(x[nt][e] - msub);
      ps += p[nt][e];
    }
  A.l_part = fmaf(A.l_part, alpha, ps);
  A.m_row = m_new;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    A.o[t][0] *= alpha;
    A.o[t][1] *= alpha;
  }
  const uint32_t a0 = pack_bf16(p[0][0], p[0][1]);
  const uint32_t a2 = pack_bf16(p[1][0], p[1][1]);
  const int mi = lane >> 3;
  const int key = rbase + 8 * (mi & 1) + (lane & 7);
#pragma unroll
  for (int dp = 0; dp < 8; ++dp) {
    const int d0 = 16 * dp;
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(swz128(vb + (d0 >> 6) * 8192, key, ((d0 & 63) >> 3) + (mi >> 1)), b0, b1, b2, b3);
    mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], a0, a2, b0, b1);
    mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], a0, a2, b2, b3);
  }
}

// ---------------------------------------------------------------------------
// Expanded spans, all on the tensor cores (query heads = M rows):
//   key part:    c = diag(sigma_K g_K) Vt_K q  (scale*log2(e) folded in),
//                kept as bf16 hi + lo A fragments (near-fp32 precision)
//   body tokens: logits = c^T U_K^T, online softmax, w += p^T U_V
//   value part:  o += diag(sigma_V g_V) w  times Vt_V (hi + lo)
// Tokens are shared among the four warps (16 per warp per 64); each warp
// keeps its own softmax state and w, so no warp waits for another.
// ---------------------------------------------------------------------------
struct ExpAcc {
  uint32_t ch[4][2];  // c hi A-fragments for k-steps of 16 ranks: {a0, a2}
  uint32_t cl[4][2];  // c lo parts
  float wacc[8][2];   // w (heads x rV) in C layout: tile jt = columns 8jt..8jt+7
  bool had;
};

__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16(x0 - hf.x, x1 - hf.y);
}

__device__ __forceinline__ void exp_key(WarpAcc& A, ExpAcc& X, const uint8_t* part, int rK,
                                        float scale_log2) {
  const int lane = threadIdx.x & 31;
  const float* sig = reinterpret_cast<const float*>(part + 16);
  const float* gat = sig + r4(rK);
  const uint32_t vt = smem_u32(part + 16 + 8 * r4(rK));
  // eight independent accumulation chains (one per 8 ranks), k-steps outside
  float cv[8][2], cw[8][2];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) cv[nt][0] = cv[nt][1] = cw[nt][0] = cw[nt][1] = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      if (8 * nt < rK) {
        uint32_t b0, b1, b2, b3;
        const int row = 8 * nt + (lane & 7), chunk = 4 * i + (lane >> 3);
        ldsm_x4(vt + row * 256 + ((chunk ^ (row & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_rows8(cv[nt][0], cv[nt][1], A.qa[2 * i][0], A.qa[2 * i][1], b0, b1);
        mma_bf16_rows8(cw[nt][0], cw[nt][1], A.qa[2 * i + 1][0], A.qa[2 * i + 1][1], b2, b3);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int j0 = 8 * nt + 2 * (lane & 3);
    cv[nt][0] = j0 < rK ? (cv[nt][0] + cw[nt][0]) * sig[j0] * gat[j0] * scale_log2 : 0.f;
    cv[nt][1] = j0 + 1 < rK ? (cv[nt][1] + cw[nt][1]) * sig[j0 + 1] * gat[j0 + 1] * scale_log2
                            : 0.f;
  }
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    split_bf16(cv[2 * ks][0], cv[2 * ks][1], X.ch[ks][0], X.cl[ks][0]);
    split_bf16(cv[2 * ks + 1][0], cv[2 * ks + 1][1], X.ch[ks][1], X.cl[ks][1]);
  }
#pragma unroll
  for (int t = 0; t < 8; ++t) X.wacc[t][0] = X.wacc[t][1] = 0.f;
  X.had = false;
}

// Body tokens [0, n) of this page; U_K rows at uk, U_V rows at uv (row
// strides r8(rK), r8(rV) bf16).  Rows or ranks past the valid ones read
// neighbouring shared memory and are masked with selects, never multiplied.
__device__ __forceinline__ void exp_tokens(WarpAcc& A, ExpAcc& X, const uint8_t* uk,
                                           const uint8_t* uv, int n, int rK, int rV, int start,
                                           int step) {
  const int lane = threadIdx.x & 31;
  const int sk = 2 * r8(rK), sv = 2 * r8(rV);  // row strides in bytes
  const uint32_t uku = smem_u32(uk), uvu = smem_u32(uv);
  const int mi = lane >> 3;
  for (int rbase = start; rbase < n; rbase += step) {
    X.had = true;
    float s[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, sl[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      if (16 * ks < rK) {
        uint32_t b0, b1, b2, b3;
        const int tok = rbase + 8 * (mi >> 1) + (lane & 7);
        ldsm_x4(uku + tok * sk + (2 * ks + (mi & 1)) * 16, b0, b1, b2, b3);
        if (16 * ks + 16 > rK) {
          const int j = 16 * ks + 2 * (lane & 3);
          const uint32_t m0 = (j < rK ? 0xffffu : 0u) | (j + 1 < rK ? 0xffff0000u : 0u);
          const uint32_t m1 = (j + 8 < rK ? 0xffffu : 0u) | (j + 9 < rK ? 0xffff0000u : 0u);
          b0 &= m0; b2 &= m0; b1 &= m1; b3 &= m1;
        }
        mma_bf16_rows8(s[0][0], s[0][1], X.ch[ks][0], X.ch[ks][1], b0, b1);
        mma_bf16_rows8(sl[0][0], sl[0][1], X.cl[ks][0], X.cl[ks][1], b0, b1);
        mma_bf16_rows8(s[1][0], s[1][1], X.ch[ks][0], X.ch[ks][1], b2, b3);
        mma_bf16_rows8(sl[1][0], sl[1][1], X.cl[ks][0], X.cl[ks][1], b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] += sl[nt][0];
      s[nt][1] += sl[nt][1];
    }
    float x[2][2], mx = kNegInf;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = rbase + 8 * nt + 2 * (lane & 3) + e;
        x[nt][e] = tok < n ? s[nt][e] : kNegInf;
        mx = fmaxf(mx, x[nt][e]);
      }
    mx = quad_max(mx);
    const float m_new = fmaxf(A.m_row, mx);
    float alpha, msub;
    softmax_rescale(A.m_row, m_new, alpha, msub);
    float p[2][2], ps = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[nt][e] = exp2f(x[nt][e] - msub);
        ps += p[nt][e];
      }
    A.l_part = fmaf(A.l_part, alpha, ps);
    A.m_row = m_new;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      A.o[t][0] *= alpha;
      A.o[t][1] *= alpha;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      X.wacc[t][0] *= alpha;
      X.wacc[t][1] *= alpha;
    }
    const uint32_t a0 = pack_bf16(p[0][0], p[0][1]);
    const uint32_t a2 = pack_bf16(p[1][0], p[1][1]);
    const bool tail = rbase + 16 > n;
    const int tk = rbase + 2 * (lane & 3);  // tokens held by b0/b2 (+8 in b1/b3)
    const uint32_t t0 = (tk < n ? 0xffffu : 0u) | (tk + 1 < n ? 0xffff0000u : 0u);
    const uint32_t t1 = (tk + 8 < n ? 0xffffu : 0u) | (tk + 9 < n ? 0xffff0000u : 0u);
#pragma unroll
    for (int jp = 0; jp < 4; ++jp) {
      if (16 * jp < rV) {
        uint32_t b0, b1, b2, b3;
        const int tok = rbase + 8 * (mi & 1) + (lane & 7);
        ldsm_x4_t(uvu + tok * sv + (2 * jp + (mi >> 1)) * 16, b0, b1, b2, b3);
        if (tail) { b0 &= t0; b2 &= t0; b1 &= t1; b3 &= t1; }
        mma_bf16_rows8(X.wacc[2 * jp][0], X.wacc[2 * jp][1], a0, a2, b0, b1);
        mma_bf16_rows8(X.wacc[2 * jp + 1][0], X.wacc[2 * jp + 1][1], a0, a2, b2, b3);
      }
    }
  }
}

__device__ __forceinline__ void exp_value(WarpAcc& A, ExpAcc& X, const uint8_t* part, int rV) {
  if (!X.had) return;
  const int lane = threadIdx.x & 31;
  const float* sig = reinterpret_cast<const float*>(part);
  const float* gat = sig + r4(rV);
  const uint32_t vt = smem_u32(part + 8 * r4(rV));
  const int mi = lane >> 3;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    if (16 * ks < rV) {
      const int j0 = 16 * ks + 2 * (lane & 3);
      float c[4];
      c[0] = j0 < rV ? X.wacc[2 * ks][0] * sig[j0] * gat[j0] : 0.f;
      c[1] = j0 + 1 < rV ? X.wacc[2 * ks][1] * sig[j0 + 1] * gat[j0 + 1] : 0.f;
      c[2] = j0 + 8 < rV ? X.wacc[2 * ks + 1][0] * sig[j0 + 8] * gat[j0 + 8] : 0.f;
      c[3] = j0 + 9 < rV ? X.wacc[2 * ks + 1][1] * sig[j0 + 9] * gat[j0 + 9] : 0.f;
      uint32_t h0, l0, h2, l2;
      split_bf16(c[0], c[1], h0, l0);
      split_bf16(c[2], c[3], h2, l2);
      const int j = 16 * ks + 8 * (mi & 1) + (lane & 7);  // Vt_V row addressed by this lane
      const bool tail = 16 * ks + 16 > rV;
      const uint32_t m0 = (j0 < rV ? 0xffffu : 0u) | (j0 + 1 < rV ? 0xffff0000u : 0u);
      const uint32_t m1 = (j0 + 8 < rV ? 0xffffu : 0u) | (j0 + 9 < rV ? 0xffff0000u : 0u);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vt + j * 256 + (((2 * dp + (mi >> 1)) ^ (j & 7)) << 4), b0, b1, b2, b3);
        if (tail) { b0 &= m0; b2 &= m0; b1 &= m1; b3 &= m1; }
        mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], h0, h2, b0, b1);
        mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], l0, l2, b0, b1);
        mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], h0, h2, b2, b3);
        mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], l0, l2, b2, b3);
      }
    }
  }
}

}  // namespace sekv
