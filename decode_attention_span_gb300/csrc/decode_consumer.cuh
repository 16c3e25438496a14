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

// One full-resolution or summary page: up to 32 rows whose 32-row boxes are
// 128B-swizzled (keys for dims 0-63 at kb, 64-127 at kb + kBoxBytes; values
// likewise at vb), folded into the warp's softmax state with one rescale.
// bias_row: for summary pages the logit bias of the page's spans (log2|S|, or
// -inf for a span that does not enter as a summary); nullptr for full rows.
// Rows >= n are masked.
__device__ __forceinline__ void consume_kv_page(WarpAcc& A, uint32_t kb, uint32_t vb, int n,
                                                const float* bias_row, float scale_log2) {
  const int lane = threadIdx.x & 31;
  const int nh = n > 16 ? 2 : 1;  // 16-row halves holding rows
  float s[2][2][2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[hh][nt][0] = s[hh][nt][1] = 0.f;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {  // 32 head dims per step
    const uint4 q = lds128(A.qfrag + (i * 32 + lane) * 16);
    const uint32_t box = kb + (i >> 1) * kBoxBytes;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if (hh < nh) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(swz128(box, 16 * hh + 8 * nt + (lane & 7), (i & 1) * 4 + (lane >> 3)), b0, b1,
                  b2, b3);
          mma_bf16_rows8(s[hh][nt][0], s[hh][nt][1], q.x, q.y, b0, b1);
          mma_bf16_rows8(s[hh][nt][0], s[hh][nt][1], q.z, q.w, b2, b3);
        }
      }
    }
  }
  float mx = kNegInf;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = 16 * hh + 8 * nt + 2 * (lane & 3) + e;
        bool valid = key < n;
        float bias = 0.f;
        if (bias_row != nullptr && valid) {
          bias = bias_row[key];
          valid = bias != kNegInf;
        }
        s[hh][nt][e] = valid ? fmaf(s[hh][nt][e], scale_log2, bias) : kNegInf;
        mx = fmaxf(mx, s[hh][nt][e]);
      }
  mx = quad_max(mx);
  const float m_new = fmaxf(A.m_row, mx);
  float alpha, msub;
  softmax_rescale(A.m_row, m_new, alpha, msub);
  float ps = 0.f;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s[hh][nt][e] = exp2f(s[hh][nt][e] - msub);
        ps += s[hh][nt][e];
      }
  A.l_part = fmaf(A.l_part, alpha, ps);
  A.m_row = m_new;
  if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      A.o[t][0] *= alpha;
      A.o[t][1] *= alpha;
    }
  }
  const int mi = lane >> 3;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    if (hh < nh) {
      const uint32_t a0 = pack_bf16(s[hh][0][0], s[hh][0][1]);
      const uint32_t a2 = pack_bf16(s[hh][1][0], s[hh][1][1]);
      const int key = 16 * hh + 8 * (mi & 1) + (lane & 7);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int d0 = 16 * dp;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(swz128(vb + (d0 >> 6) * kBoxBytes, key, ((d0 & 63) >> 3) + (mi >> 1)), b0, b1,
                  b2, b3);
        mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], a0, a2, b0, b1);
        mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], a0, a2, b2, b3);
      }
    }
  }
}

// Routing logits z[span][head] = s_span . y_head of a routing page (two
// 128B-swizzled boxes of 64 rows x 32 floats) on the tensor cores: spans are
// the M rows, heads the N columns, routing dims K; s and y both split into
// bf16 hi + lo parts (hi*hi + hi*lo + lo*hi, error about 2^-16 of sum |s_d y_d|).
// Returns the 64-bit mask of spans with z > theta for some head of the group.
__device__ __forceinline__ unsigned long long route_hits(const uint8_t* page, int n,
                                                        const float* ys, const float* theta,
                                                        int G) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  uint32_t bh[4][2], bl[4][2];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const float2 v = *reinterpret_cast<const float2*>(ys + gid * kRouteDim + 16 * ks + 8 * hf +
                                                        2 * tig);
      split_bf16(v.x, v.y, bh[ks][hf], bl[ks][hf]);
    }
  const bool ok0 = 2 * tig < G, ok1 = 2 * tig + 1 < G;
  const float th0 = theta[2 * tig], th1 = theta[2 * tig + 1];
  unsigned long long hits = 0;
#pragma unroll 1
  for (int mt = 0; 16 * mt < n; ++mt) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t ah[4], al[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int row = 16 * mt + gid + 8 * (q & 1);
        const int dim = 16 * ks + 2 * tig + 8 * (q >> 1);
        const float2 v = *reinterpret_cast<const float2*>(
            page + (dim >> 5) * 8192 + row * 128 + ((((dim & 31) >> 2) ^ (row & 7)) << 4) +
            (dim & 3) * 4);
        split_bf16(v.x, v.y, ah[q], al[q]);
      }
      mma_bf16_16816(acc, ah[0], ah[1], ah[2], ah[3], bh[ks][0], bh[ks][1]);
      mma_bf16_16816(acc, ah[0], ah[1], ah[2], ah[3], bl[ks][0], bl[ks][1]);
      mma_bf16_16816(acc, al[0], al[1], al[2], al[3], bh[ks][0], bh[ks][1]);
    }
    // rows gid, gid + 8; heads 2 tig, 2 tig + 1; any head of the quad
    const bool hA = (ok0 && acc[0] > th0) || (ok1 && acc[1] > th1);
    const bool hB = (ok0 && acc[2] > th0) || (ok1 && acc[3] > th1);
    const uint32_t bA = __ballot_sync(0xffffffffu, hA), bB = __ballot_sync(0xffffffffu, hB);
    uint32_t m16 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      m16 |= (((bA >> (4 * i)) & 0xFu) ? 1u : 0u) << i;
      m16 |= (((bB >> (4 * i)) & 0xFu) ? 1u : 0u) << (i + 8);
    }
    hits |= (unsigned long long)m16 << (16 * mt);
  }
  return hits;
}

// ---------------------------------------------------------------------------
// Expanded spans, all on the tensor cores (query heads = M rows):
//   key part:    c = diag(sigma_K g_K) Vt_K q  (scale*log2(e) folded in),
//                kept as bf16 hi + lo A fragments (near-fp32 precision)
//   body tokens: logits = c^T U_K^T, online softmax, w += p^T U_V
//   value part:  o += diag(sigma_V g_V) w  times Vt_V (hi + lo)
// One warp handles a whole record.
// ---------------------------------------------------------------------------
struct ExpAcc {
  uint32_t ch[4][2];  // c hi A-fragments for k-steps of 16 ranks: {a0, a2}
  uint32_t cl[4][2];  // c lo parts
  float wacc[8][2];   // w (heads x rV) in C layout: tile jt = columns 8jt..8jt+7
  bool had;
};

__device__ __forceinline__ void exp_key(const WarpAcc& A, ExpAcc& X, const uint8_t* part, int rK,
                                        float scale_log2) {
  const int lane = threadIdx.x & 31;
  const float* sig = reinterpret_cast<const float*>(part + 16);
  const float* gat = sig + r4(rK);
  const uint32_t vt = smem_u32(part + 16 + 8 * r4(rK));
  float cv[8][2];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) cv[nt][0] = cv[nt][1] = 0.f;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {  // 32 head dims per step
    const uint4 q = lds128(A.qfrag + (i * 32 + lane) * 16);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      if (8 * nt < rK) {
        uint32_t b0, b1, b2, b3;
        const int row = 8 * nt + (lane & 7), chunk = 4 * i + (lane >> 3);
        ldsm_x4(vt + row * 256 + ((chunk ^ (row & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_rows8(cv[nt][0], cv[nt][1], q.x, q.y, b0, b1);
        mma_bf16_rows8(cv[nt][0], cv[nt][1], q.z, q.w, b2, b3);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int j0 = 8 * nt + 2 * (lane & 3);
    cv[nt][0] = j0 < rK ? cv[nt][0] * sig[j0] * gat[j0] * scale_log2 : 0.f;
    cv[nt][1] = j0 + 1 < rK ? cv[nt][1] * sig[j0 + 1] * gat[j0 + 1] * scale_log2 : 0.f;
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
// strides r8(rK), r8(rV) bf16).  Tokens go in blocks of 32: the two 16-token
// score tiles are independent, then one softmax rescale per block.  Rows or
// ranks past the valid ones read neighbouring shared memory and are masked
// with selects, never multiplied.
__device__ __forceinline__ void exp_tokens(WarpAcc& A, ExpAcc& X, const uint8_t* uk,
                                           const uint8_t* uv, int n, int rK, int rV) {
  const int lane = threadIdx.x & 31;
  const int sk = 2 * r8(rK), sv = 2 * r8(rV);  // row strides in bytes
  const uint32_t uku = smem_u32(uk), uvu = smem_u32(uv);
  const int mi = lane >> 3;
  // rank-tail masks of the last k-step of U_K
  const int jr = 16 * ((rK - 1) >> 4) + 2 * (lane & 3);
  const uint32_t rm0 = (jr < rK ? 0xffffu : 0u) | (jr + 1 < rK ? 0xffff0000u : 0u);
  const uint32_t rm1 = (jr + 8 < rK ? 0xffffu : 0u) | (jr + 9 < rK ? 0xffff0000u : 0u);
#pragma unroll 1
  for (int rb = 0; rb < n; rb += 32) {
    X.had = true;
    const int nch = (n - rb) > 16 ? 2 : 1;
    float s[2][2][2];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) s[ch][nt][0] = s[ch][nt][1] = 0.f;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      if (ch < nch) {
        const int tok = rb + 16 * ch + 8 * (mi >> 1) + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          if (16 * ks < rK) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(uku + tok * sk + (2 * ks + (mi & 1)) * 16, b0, b1, b2, b3);
            if (16 * ks + 16 > rK) {
              b0 &= rm0; b2 &= rm0; b1 &= rm1; b3 &= rm1;
            }
            mma_bf16_rows8(s[ch][0][0], s[ch][0][1], X.ch[ks][0], X.ch[ks][1], b0, b1);
            mma_bf16_rows8(s[ch][1][0], s[ch][1][1], X.ch[ks][0], X.ch[ks][1], b2, b3);
            mma_bf16_rows8(s[ch][0][0], s[ch][0][1], X.cl[ks][0], X.cl[ks][1], b0, b1);
            mma_bf16_rows8(s[ch][1][0], s[ch][1][1], X.cl[ks][0], X.cl[ks][1], b2, b3);
          }
        }
      }
    }
    float mx = kNegInf;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = rb + 16 * ch + 8 * nt + 2 * (lane & 3) + e;
          s[ch][nt][e] = tok < n ? s[ch][nt][e] : kNegInf;
          mx = fmaxf(mx, s[ch][nt][e]);
        }
    mx = quad_max(mx);
    const float m_new = fmaxf(A.m_row, mx);
    float alpha, msub;
    softmax_rescale(A.m_row, m_new, alpha, msub);
    float ps = 0.f;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[ch][nt][e] = exp2f(s[ch][nt][e] - msub);
          ps += s[ch][nt][e];
        }
    A.l_part = fmaf(A.l_part, alpha, ps);
    A.m_row = m_new;
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
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
    }
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      if (ch < nch) {
        const int rbase = rb + 16 * ch;
        const uint32_t a0 = pack_bf16(s[ch][0][0], s[ch][0][1]);
        const uint32_t a2 = pack_bf16(s[ch][1][0], s[ch][1][1]);
        const bool tail = rbase + 16 > n;
        const int tk = rbase + 2 * (lane & 3);  // tokens held by b0/b2 (+8 in b1/b3)
        const uint32_t t0 = (tk < n ? 0xffffu : 0u) | (tk + 1 < n ? 0xffff0000u : 0u);
        const uint32_t t1 = (tk + 8 < n ? 0xffffu : 0u) | (tk + 9 < n ? 0xffff0000u : 0u);
        const int tok = rbase + 8 * (mi & 1) + (lane & 7);
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          if (16 * jp < rV) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(uvu + tok * sv + (2 * jp + (mi >> 1)) * 16, b0, b1, b2, b3);
            if (tail) { b0 &= t0; b2 &= t0; b1 &= t1; b3 &= t1; }
            mma_bf16_rows8(X.wacc[2 * jp][0], X.wacc[2 * jp][1], a0, a2, b0, b1);
            mma_bf16_rows8(X.wacc[2 * jp + 1][0], X.wacc[2 * jp + 1][1], a0, a2, b2, b3);
          }
        }
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
  // coefficient A fragments of every k-step of 16 ranks, hi and lo; the
  // rolled loop below always uses index 0 and shifts the rest down
  uint32_t h0[4], h2[4], l0[4], l2[4];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const int j0 = 16 * ks + 2 * (lane & 3);
    const float c0 = j0 < rV ? X.wacc[2 * ks][0] * sig[j0] * gat[j0] : 0.f;
    const float c1 = j0 + 1 < rV ? X.wacc[2 * ks][1] * sig[j0 + 1] * gat[j0 + 1] : 0.f;
    const float c2 = j0 + 8 < rV ? X.wacc[2 * ks + 1][0] * sig[j0 + 8] * gat[j0 + 8] : 0.f;
    const float c3 = j0 + 9 < rV ? X.wacc[2 * ks + 1][1] * sig[j0 + 9] * gat[j0 + 9] : 0.f;
    split_bf16(c0, c1, h0[ks], l0[ks]);
    split_bf16(c2, c3, h2[ks], l2[ks]);
  }
  // rank-tail masks of the last k-step of Vt_V rows
  const int jr = 16 * ((rV - 1) >> 4) + 2 * (lane & 3);
  const uint32_t m0 = (jr < rV ? 0xffffu : 0u) | (jr + 1 < rV ? 0xffff0000u : 0u);
  const uint32_t m1 = (jr + 8 < rV ? 0xffffu : 0u) | (jr + 9 < rV ? 0xffff0000u : 0u);
#pragma unroll 1
  for (int ks = 0; 16 * ks < rV; ++ks) {
    const int j = 16 * ks + 8 * (mi & 1) + (lane & 7);  // Vt_V row addressed by this lane
    const bool tail = 16 * ks + 16 > rV;
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vt + j * 256 + (((2 * dp + (mi >> 1)) ^ (j & 7)) << 4), b0, b1, b2, b3);
      if (tail) { b0 &= m0; b2 &= m0; b1 &= m1; b3 &= m1; }
      mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], h0[0], h2[0], b0, b1);
      mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], h0[0], h2[0], b2, b3);
      mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], l0[0], l2[0], b0, b1);
      mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], l0[0], l2[0], b2, b3);
    }
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      h0[t] = h0[t + 1];
      h2[t] = h2[t + 1];
      l0[t] = l0[t + 1];
      l2[t] = l2[t + 1];
    }
  }
}

}  // namespace sekv
