// Consumer math of the decode kernel: the routing logits and the online
// softmax over full-resolution rows, summary rows and expanded records.
//
// Every product runs on mma.sync m16n8k16 (bf16 in, fp32 accumulate) in
// transposed form: keys, tokens, ranks or head dims are the 16 M rows and
// the query heads of the GQA group (at most 8) are the N columns, so no
// tile row is wasted.  A lane (g = lane / 4, q = lane % 4) holds, of an
// M x 8 result tile, rows g and g + 8 of columns (heads) 2q and 2q + 1.
// Probabilities and coefficients produced in that layout become the B
// operand of the next product through movmatrix (an 8 x 8 transpose in
// registers).  The query's B fragments sit in shared memory (qfrag).
#pragma once

#include "decode_attn.cuh"

namespace sekv {

constexpr float kNegInf = -__builtin_huge_valf();

struct WarpAcc {
  float o[8][4];   // O^T tiles: tile t holds dims 16 t + g (c0: head 2q, c1: head 2q + 1)
                   // and 16 t + g + 8 (c2: head 2q, c3: head 2q + 1)
  float m[2];      // running max of heads 2q, 2q + 1 (log2 domain; equal in a column)
  float l[2];      // this lane's share of the sums of heads 2q, 2q + 1
  uint32_t qfrag;  // shared address of the query's B fragments (4 x 32 lanes x 16 B)
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

// D = A * B + D, one m16n8k16 bf16 tile with fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8 x 8 matrix of bf16 pairs held one row-pair per lane.
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// max / sum over the eight lanes that share a column pair (same lane % 4)
__device__ __forceinline__ float col_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}
__device__ __forceinline__ float col_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  return v + __shfl_xor_sync(0xffffffffu, v, 16);
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

// Lazy online-softmax re-basing: the running max m of a head only moves when
// a new logit exceeds it by more than kRebase (log2 units), so exponentials
// stay below 2^kRebase and most tiles skip the reductions and the rescale.
// The output is normalised by the sum taken against the same m, so the
// choice of m changes only rounding.
constexpr float kRebase = 8.f;

__device__ __forceinline__ float rescale_factor(float m_old, float m_new) {
  return m_new == kNegInf ? 1.f : exp2f(m_old - m_new);
}

// Re-base the warp's state to cover this lane's tile maxima mx0, mx1 (heads
// 2q, 2q + 1) if some lane's exceeds the running max by more than kRebase;
// returns the two rescale factors (1 when nothing moved).
__device__ __forceinline__ float2 rebase_if_needed(WarpAcc& A, float mx0, float mx1) {
  float2 alpha = make_float2(1.f, 1.f);
  if (__any_sync(0xffffffffu, mx0 > A.m[0] + kRebase || mx1 > A.m[1] + kRebase)) {
    const float n0 = fmaxf(A.m[0], col_max(mx0)), n1 = fmaxf(A.m[1], col_max(mx1));
    alpha.x = rescale_factor(A.m[0], n0);
    alpha.y = rescale_factor(A.m[1], n1);
    A.m[0] = n0;
    A.m[1] = n1;
    A.l[0] *= alpha.x;
    A.l[1] *= alpha.y;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      A.o[t][0] *= alpha.x;
      A.o[t][1] *= alpha.y;
      A.o[t][2] *= alpha.x;
      A.o[t][3] *= alpha.y;
    }
  }
  return alpha;
}

// Probabilities of a 16 x 8 score tile s (rows g, g + 8; heads 2q, 2q + 1)
// against the running max, added into the sums, and returned as the B
// fragments (rows = keys/tokens, columns = heads) of the following product.
__device__ __forceinline__ void probs_to_b(WarpAcc& A, float (&s)[4], uint32_t& b0,
                                           uint32_t& b1) {
  const float m0 = A.m[0] == kNegInf ? 0.f : A.m[0];
  const float m1 = A.m[1] == kNegInf ? 0.f : A.m[1];
  s[0] = ex2_approx(s[0] - m0);
  s[1] = ex2_approx(s[1] - m1);
  s[2] = ex2_approx(s[2] - m0);
  s[3] = ex2_approx(s[3] - m1);
  A.l[0] += s[0] + s[2];
  A.l[1] += s[1] + s[3];
  b0 = movtrans(pack_bf16(s[0], s[1]));
  b1 = movtrans(pack_bf16(s[2], s[3]));
}

// Masks of the bf16 pairs at k indices j, j + 1 (m0) and j + 8, j + 9 (m1),
// j = base + 2q, against a count (keys, tokens or ranks past it read as 0).
__device__ __forceinline__ void pair_masks(int base, int count, uint32_t& m0, uint32_t& m1) {
  const int j = base + 2 * (threadIdx.x & 3);
  m0 = (j < count ? 0xffffu : 0u) | (j + 1 < count ? 0xffff0000u : 0u);
  m1 = (j + 8 < count ? 0xffffu : 0u) | (j + 9 < count ? 0xffff0000u : 0u);
}

// One tile of 16 full-resolution or summary rows whose two 128-byte halves
// sit in 128B-swizzled boxes `half` bytes apart (keys: dims 0-63 at kb,
// 64-127 at kb + half; values likewise at vb; kb and vb point at the tile's
// first row, and a box's swizzle runs on in its later rows), folded into the
// warp's softmax state with at most one rescale.  bias_row: for summary pages
// the logit bias of the page's spans (log2|S|, or -inf for a span that does
// not enter as a summary); nullptr for full rows.  Rows >= n are masked.
//   S^T (16 keys x 8 heads) = K (16 x 128) q^T, then O^T += V^T P^T.
template <bool MQ>
__device__ __forceinline__ void consume_rows16(WarpAcc& A, uint32_t kb, uint32_t vb, int n,
                                               const float* bias_row, float scale_log2,
                                               int half, const uint8_t* cmask_row) {
  const int lane = threadIdx.x & 31, g = lane >> 2, mi = lane >> 3;
  // four accumulator chains (k-steps 4 j + 0..3), added at the end
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  float s2[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
  const int krow = (lane & 7) + 8 * (mi & 1);
#pragma unroll 1
  for (int i = 0; i < 4; i += 2) {  // head dims 32 i .. 32 i + 63: the box of half i / 2
    const uint4 qv = lds128(A.qfrag + (i * 32 + lane) * 16);
    const uint4 qw = lds128(A.qfrag + ((i + 1) * 32 + lane) * 16);
    const uint32_t box = kb + (i >> 1) * half;
    uint32_t a0, a1, a2, a3;
    ldsm_x4(swz128(box, krow, (mi >> 1)), a0, a1, a2, a3);
    mma16816(s0, a0, a1, a2, a3, qv.x, qv.y);
    ldsm_x4(swz128(box, krow, 2 + (mi >> 1)), a0, a1, a2, a3);
    mma16816(s1, a0, a1, a2, a3, qv.z, qv.w);
    ldsm_x4(swz128(box, krow, 4 + (mi >> 1)), a0, a1, a2, a3);
    mma16816(s2, a0, a1, a2, a3, qw.x, qw.y);
    ldsm_x4(swz128(box, krow, 6 + (mi >> 1)), a0, a1, a2, a3);
    mma16816(s3, a0, a1, a2, a3, qw.z, qw.w);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    s0[e] += s2[e];
    s1[e] += s3[e];
  }
  float s[4];
  float bias0 = 0.f, bias1 = 0.f;
  bool v0 = g < n, v1 = g + 8 < n;
  if (bias_row != nullptr) {
    bias0 = v0 ? bias_row[g] : kNegInf;
    bias1 = v1 ? bias_row[g + 8] : kNegInf;
    v0 = v0 && bias0 != kNegInf;
    v1 = v1 && bias1 != kNegInf;
  }
  s[0] = v0 ? fmaf(s0[0] + s1[0], scale_log2, bias0) : kNegInf;
  s[1] = v0 ? fmaf(s0[1] + s1[1], scale_log2, bias0) : kNegInf;
  s[2] = v1 ? fmaf(s0[2] + s1[2], scale_log2, bias1) : kNegInf;
  s[3] = v1 ? fmaf(s0[3] + s1[3], scale_log2, bias1) : kNegInf;
  if (MQ) {
    // multi-query decode: a summary row is not seen by the columns (query
    // tokens) that expand its span
    const int c0 = 2 * (lane & 3);
    const unsigned m0 = v0 ? cmask_row[g] : 0u, m1 = v1 ? cmask_row[g + 8] : 0u;
    if ((m0 >> c0) & 1u) s[0] = kNegInf;
    if ((m0 >> (c0 + 1)) & 1u) s[1] = kNegInf;
    if ((m1 >> c0) & 1u) s[2] = kNegInf;
    if ((m1 >> (c0 + 1)) & 1u) s[3] = kNegInf;
  }
  rebase_if_needed(A, fmaxf(s[0], s[2]), fmaxf(s[1], s[3]));
  uint32_t b0, b1;
  probs_to_b(A, s, b0, b1);
  // value rows past n (zero fill or unrelated rows) must not reach o
  uint32_t t0, t1;
  pair_masks(0, n, t0, t1);
  const int vrow = (lane & 7) + 8 * (mi >> 1);
#pragma unroll
  for (int dt = 0; dt < 8; ++dt) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(swz128(vb + (dt >> 2) * half, vrow, 2 * (dt & 3) + (mi & 1)), a0, a1, a2, a3);
    a0 &= t0; a1 &= t0; a2 &= t1; a3 &= t1;
    mma16816(A.o[dt], a0, a1, a2, a3, b0, b1);
  }
}

// A page of 32 full-resolution rows (two 16-row tiles, laid out as for
// consume_rows16, the second 16 rows after the first), folded into the
// warp's softmax state at once: the two tiles' logit products run as
// independent chains, and the page takes at most one rescale.  Rows >= n are
// masked.
__device__ __forceinline__ void consume_rows32(WarpAcc& A, uint32_t kb, uint32_t vb, int n,
                                               float scale_log2, int half) {
  const int lane = threadIdx.x & 31, g = lane >> 2, mi = lane >> 3;
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};  // rows 0-15
  float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};  // rows 16-31
  const int krow = (lane & 7) + 8 * (mi & 1);
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {  // head dims 32 i .. 32 i + 31: k-steps 2 i, 2 i + 1
    const uint4 qv = lds128(A.qfrag + (i * 32 + lane) * 16);
    const uint32_t box = kb + (i >> 1) * half;
    uint32_t a0, a1, a2, a3;
    ldsm_x4(swz128(box, krow, 4 * (i & 1) + (mi >> 1)), a0, a1, a2, a3);
    mma16816(s0, a0, a1, a2, a3, qv.x, qv.y);
    ldsm_x4(swz128(box, krow + 16, 4 * (i & 1) + (mi >> 1)), a0, a1, a2, a3);
    mma16816(u0, a0, a1, a2, a3, qv.x, qv.y);
    ldsm_x4(swz128(box, krow, 4 * (i & 1) + 2 + (mi >> 1)), a0, a1, a2, a3);
    mma16816(s1, a0, a1, a2, a3, qv.z, qv.w);
    ldsm_x4(swz128(box, krow + 16, 4 * (i & 1) + 2 + (mi >> 1)), a0, a1, a2, a3);
    mma16816(u1, a0, a1, a2, a3, qv.z, qv.w);
  }
  const bool v0 = g < n, v1 = g + 8 < n, v2 = g + 16 < n, v3 = g + 24 < n;
  float s[4], u[4];
  s[0] = v0 ? (s0[0] + s1[0]) * scale_log2 : kNegInf;
  s[1] = v0 ? (s0[1] + s1[1]) * scale_log2 : kNegInf;
  s[2] = v1 ? (s0[2] + s1[2]) * scale_log2 : kNegInf;
  s[3] = v1 ? (s0[3] + s1[3]) * scale_log2 : kNegInf;
  u[0] = v2 ? (u0[0] + u1[0]) * scale_log2 : kNegInf;
  u[1] = v2 ? (u0[1] + u1[1]) * scale_log2 : kNegInf;
  u[2] = v3 ? (u0[2] + u1[2]) * scale_log2 : kNegInf;
  u[3] = v3 ? (u0[3] + u1[3]) * scale_log2 : kNegInf;
  rebase_if_needed(A, fmaxf(fmaxf(s[0], s[2]), fmaxf(u[0], u[2])),
                   fmaxf(fmaxf(s[1], s[3]), fmaxf(u[1], u[3])));
  uint32_t b0, b1, c0, c1;
  probs_to_b(A, s, b0, b1);
  probs_to_b(A, u, c0, c1);
  // value rows past n (zero fill or unrelated rows) must not reach o
  uint32_t t0, t1, t2, t3;
  pair_masks(0, n, t0, t1);
  pair_masks(16, n, t2, t3);
  const int vrow = (lane & 7) + 8 * (mi >> 1);
#pragma unroll
  for (int dt = 0; dt < 8; ++dt) {
    const uint32_t vbox = vb + (dt >> 2) * half;
    const int chunk = 2 * (dt & 3) + (mi & 1);
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(swz128(vbox, vrow, chunk), a0, a1, a2, a3);
    a0 &= t0; a1 &= t0; a2 &= t1; a3 &= t1;
    mma16816(A.o[dt], a0, a1, a2, a3, b0, b1);
    ldsm_x4_t(swz128(vbox, vrow + 16, chunk), a0, a1, a2, a3);
    a0 &= t2; a1 &= t2; a2 &= t3; a3 &= t3;
    mma16816(A.o[dt], a0, a1, a2, a3, c0, c1);
  }
}

// Routing logits z[span][head] = s_span . y_head of a routing page (two
// 128B-swizzled boxes of 32 rows x 32 floats: routing dims 0-31, then 32-63)
// in fp32 FMAs, lane l taking span l, four heads per pass (y rows past the
// group are zero and ignored).  Chunk c of a row sits at c ^ (row & 7), so
// eight lanes read eight different bank groups; the y reads are broadcasts.
// Returns whether some head h of the group has z > theta_h for this lane's
// span (rows past the page's spans are computed and ignored by the caller).
__device__ __forceinline__ unsigned route32(const uint8_t* page, const float* ys,
                                            const float* theta, int G) {
  const int lane = threadIdx.x & 31, sw = lane & 7;
  unsigned hit = 0u;  // bit h: column h's logit passes its threshold
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
      if (h0 + hh < G && z[hh] > theta[h0 + hh]) hit |= 1u << (h0 + hh);
  }
  return hit;
}

// ---------------------------------------------------------------------------
// Expanded spans (one warp per record), in factor space:
//   key part:    c^T (ranks x heads) = diag(sigma_K g_K) Vt_K q^T, scale*log2(e)
//                folded in, kept as bf16 hi + lo B fragments (near-fp32)
//   body tokens: S^T = U_K c (tokens x heads), softmax, w^T += U_V^T P^T
//   value part:  O^T += Vt_V^T diag(sigma_V g_V) w^T (hi + lo)
// KS = rank k-steps of 16 (ranks up to 16 KS): every loop has a fixed trip
// count; ranks past the record's own are masked arithmetically (no
// data-dependent branches in the inner loops).
// ---------------------------------------------------------------------------
template <int KS>
struct ExpAcc {
  uint32_t ch[KS][2];  // c hi B fragments, k-step = ranks 16 ks .. 16 ks + 15
  uint32_t cl[KS][2];  // c lo parts
  float w[KS][4];      // w^T tiles (ranks 16 T + g, + 8; heads 2q, 2q + 1)
  bool had;
};

template <int KS>
__device__ __forceinline__ void exp_key(const WarpAcc& A, ExpAcc<KS>& X, const uint8_t* part,
                                        int rK, float scale_log2) {
  const int lane = threadIdx.x & 31, g = lane >> 2, mi = lane >> 3;
  const float* sig = reinterpret_cast<const float*>(part + 16);
  const float* gat = sig + r4(rK);
  const uint32_t vt = smem_u32(part + 16 + 8 * r4(rK));
  // two accumulator chains per rank tile (the two 16-dim halves of each
  // 32-dim step), added at the end
  float cv[KS][4], cw[KS][4];
#pragma unroll
  for (int t = 0; t < KS; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) cv[t][e] = cw[t][e] = 0.f;
  // Vt_K rows past rK read the record's next bytes; their rows of c are
  // dropped by the selects below
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // head dims 32 i .. 32 i + 31
    const uint4 qv = lds128(A.qfrag + (i * 32 + lane) * 16);
#pragma unroll
    for (int t = 0; t < KS; ++t) {
      const int row = 16 * t + (lane & 7) + 8 * (mi & 1);
      uint32_t a0, a1, a2, a3;
      ldsm_x4(vt + row * 256 + (((4 * i + (mi >> 1)) ^ (row & 7)) << 4), a0, a1, a2, a3);
      mma16816(cv[t], a0, a1, a2, a3, qv.x, qv.y);
      ldsm_x4(vt + row * 256 + (((4 * i + 2 + (mi >> 1)) ^ (row & 7)) << 4), a0, a1, a2, a3);
      mma16816(cw[t], a0, a1, a2, a3, qv.z, qv.w);
    }
  }
#pragma unroll
  for (int t = 0; t < KS; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) cv[t][e] += cw[t][e];
#pragma unroll
  for (int t = 0; t < KS; ++t) {
    const int r0 = 16 * t + g, r1 = r0 + 8;
    const float f0 = r0 < rK ? sig[r0] * gat[r0] * scale_log2 : 0.f;
    const float f1 = r1 < rK ? sig[r1] * gat[r1] * scale_log2 : 0.f;
    const float c0 = r0 < rK ? cv[t][0] * f0 : 0.f, c1 = r0 < rK ? cv[t][1] * f0 : 0.f;
    const float c2 = r1 < rK ? cv[t][2] * f1 : 0.f, c3 = r1 < rK ? cv[t][3] * f1 : 0.f;
    uint32_t h01, l01, h23, l23;
    split_bf16(c0, c1, h01, l01);
    split_bf16(c2, c3, h23, l23);
    X.ch[t][0] = movtrans(h01);
    X.ch[t][1] = movtrans(h23);
    X.cl[t][0] = movtrans(l01);
    X.cl[t][1] = movtrans(l23);
    X.w[t][0] = X.w[t][1] = X.w[t][2] = X.w[t][3] = 0.f;
  }
  X.had = false;
}

// NT (1 or 2) tiles of 16 body tokens from token rb on: logits U_K c (the
// hi and lo products of c in separate chains, the tiles' chains interleaved),
// one re-basing check over the tiles, then w^T += U_V^T P^T.  Tokens >= n
// are masked; so are the columns (query tokens) outside cm in multi-query
// decode.
template <int KS, bool MQ, int NT>
__device__ __forceinline__ void tok_tiles(WarpAcc& A, ExpAcc<KS>& X, uint32_t uku, uint32_t uvu,
                                          int rb, int n, int rK, int sk, int sv, int wk, int wv,
                                          unsigned cm) {
  const int lane = threadIdx.x & 31, g = lane >> 2, mi = lane >> 3;
  float s[NT][4], sl[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[j][e] = sl[j][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t m0, m1;
    pair_masks(16 * ks, rK, m0, m1);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int tq = rb + 16 * j + (lane & 7) + 8 * (mi & 1);
      uint32_t a0, a1, a2, a3;
      ldsm_x4(uku + tq * sk + (((2 * ks + (mi >> 1)) ^ u_swz(tq, wk)) << 4), a0, a1, a2, a3);
      a0 &= m0; a1 &= m0; a2 &= m1; a3 &= m1;
      mma16816(s[j], a0, a1, a2, a3, X.ch[ks][0], X.ch[ks][1]);
      mma16816(sl[j], a0, a1, a2, a3, X.cl[ks][0], X.cl[ks][1]);
    }
  }
  float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) s[j][e] += sl[j][e];
    if (rb + 16 * j + g >= n) s[j][0] = s[j][1] = kNegInf;
    if (rb + 16 * j + g + 8 >= n) s[j][2] = s[j][3] = kNegInf;
    if (MQ) {
      if (!((cm >> (2 * (lane & 3))) & 1u)) s[j][0] = s[j][2] = kNegInf;
      if (!((cm >> (2 * (lane & 3) + 1)) & 1u)) s[j][1] = s[j][3] = kNegInf;
    }
    mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][2]));
    mx1 = fmaxf(mx1, fmaxf(s[j][1], s[j][3]));
  }
  const float2 alpha = rebase_if_needed(A, mx0, mx1);
  if (alpha.x != 1.f || alpha.y != 1.f) {
#pragma unroll
    for (int t = 0; t < KS; ++t) {
      X.w[t][0] *= alpha.x;
      X.w[t][1] *= alpha.y;
      X.w[t][2] *= alpha.x;
      X.w[t][3] *= alpha.y;
    }
  }
  uint32_t b[NT][2], tm[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    probs_to_b(A, s[j], b[j][0], b[j][1]);
    pair_masks(rb + 16 * j, n, tm[j][0], tm[j][1]);
  }
#pragma unroll
  for (int t = 0; t < KS; ++t) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int tv = rb + 16 * j + (lane & 7) + 8 * (mi >> 1);
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(uvu + tv * sv + (((2 * t + (mi & 1)) ^ u_swz(tv, wv)) << 4), a0, a1, a2, a3);
      a0 &= tm[j][0]; a1 &= tm[j][0]; a2 &= tm[j][1]; a3 &= tm[j][1];
      mma16816(X.w[t], a0, a1, a2, a3, b[j][0], b[j][1]);
    }
  }
}

// Body tokens [0, n) of this page; U_K rows at uk, U_V rows at uv (row
// strides r8(rK), r8(rV) bf16, chunks swizzled by u_swz: a page starts at a
// token that is a multiple of 16), in pairs of 16-token tiles with lazy
// re-basing, the last tile alone if it is odd.  Rows or ranks past the valid
// ones read neighbouring shared memory (up to 31 rows past a block's end) and
// are masked, never multiplied.
template <int KS, bool MQ>
__device__ __forceinline__ void exp_tokens(WarpAcc& A, ExpAcc<KS>& X, const uint8_t* uk,
                                           const uint8_t* uv, int n, int rK, int rV,
                                           unsigned cm) {
  if (n <= 0) return;
  const int sk = 2 * r8(rK), sv = 2 * r8(rV);  // row strides in bytes
  const int wk = r8(rK) >> 3, wv = r8(rV) >> 3;  // 16-byte chunks per row (swizzled)
  const uint32_t uku = smem_u32(uk), uvu = smem_u32(uv);
  X.had = true;
  int rb = 0;
#pragma unroll 1
  for (; rb + 16 < n; rb += 32) tok_tiles<KS, MQ, 2>(A, X, uku, uvu, rb, n, rK, sk, sv, wk, wv, cm);
  if (rb < n) tok_tiles<KS, MQ, 1>(A, X, uku, uvu, rb, n, rK, sk, sv, wk, wv, cm);
}

template <int KS>
__device__ __forceinline__ void exp_value(WarpAcc& A, ExpAcc<KS>& X, const uint8_t* part,
                                          int rV) {
  if (!X.had) return;
  const int lane = threadIdx.x & 31, g = lane >> 2, mi = lane >> 3;
  const float* sig = reinterpret_cast<const float*>(part);
  const float* gat = sig + r4(rV);
  const uint32_t vt = smem_u32(part + 8 * r4(rV));
#pragma unroll
  for (int t = 0; t < KS; ++t) {
    // coefficients diag(sigma_V g_V) w^T of ranks 16 t .. 16 t + 15 as B
    // fragments, hi and lo
    const int r0 = 16 * t + g, r1 = r0 + 8;
    const float f0 = r0 < rV ? sig[r0] * gat[r0] : 0.f;
    const float f1 = r1 < rV ? sig[r1] * gat[r1] : 0.f;
    const float c0 = r0 < rV ? X.w[t][0] * f0 : 0.f, c1 = r0 < rV ? X.w[t][1] * f0 : 0.f;
    const float c2 = r1 < rV ? X.w[t][2] * f1 : 0.f, c3 = r1 < rV ? X.w[t][3] * f1 : 0.f;
    uint32_t h01, l01, h23, l23, m0, m1;
    split_bf16(c0, c1, h01, l01);
    split_bf16(c2, c3, h23, l23);
    const uint32_t bh0 = movtrans(h01), bh1 = movtrans(h23);
    const uint32_t bl0 = movtrans(l01), bl1 = movtrans(l23);
    pair_masks(16 * t, rV, m0, m1);
    const int row = 16 * t + (lane & 7) + 8 * (mi >> 1);  // Vt_V row (rank) of this lane
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
      uint32_t a0, a1, a2, a3;
      const int chunk = 2 * dt + (mi & 1);
      ldsm_x4_t(vt + row * 256 + ((chunk ^ (row & 7)) << 4), a0, a1, a2, a3);
      a0 &= m0; a1 &= m0; a2 &= m1; a3 &= m1;
      mma16816(A.o[dt], a0, a1, a2, a3, bh0, bh1);
      mma16816(A.o[dt], a0, a1, a2, a3, bl0, bl1);
    }
  }
}

}  // namespace sekv
