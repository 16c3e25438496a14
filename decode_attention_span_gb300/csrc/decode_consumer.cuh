// Consumer warps of the decode kernel: routing and the online softmax.
#pragma once

#include "decode_attn.cuh"

namespace sekv {

constexpr float kNegInf = -__builtin_huge_valf();

struct WarpAcc {
  float o[16][2];   // output accumulator, row r0 = lane/4, dims 8t + 2(lane%4) + {0,1}
  float m_row;      // running max of row r0 (log2 domain)
  float l_part;     // this lane's share of the row sum
  float w[8][2];    // expanded span: U_V^T p for head h, columns lane and lane+32
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
// at +8192), vb likewise for values.  info: span info of the page's first
// row for summary pages (nullptr for full rows).
__device__ __forceinline__ void consume_kv_tile(WarpAcc& A, uint32_t kb, uint32_t vb, int n,
                                                const uint16_t* info, float scale_log2) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int rbase = 16 * w;
  if (rbase >= n) return;
  float s[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t box = kb + (i >> 1) * 8192;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(swz128(box, rbase + 8 * nt + (lane & 7), (i & 1) * 4 + (lane >> 3)), b0, b1, b2,
              b3);
      mma_bf16_rows8(s[nt][0], s[nt][1], A.qa[2 * i][0], A.qa[2 * i][1], b0, b1);
      mma_bf16_rows8(s[nt][0], s[nt][1], A.qa[2 * i + 1][0], A.qa[2 * i + 1][1], b2, b3);
    }
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
      if (info != nullptr && valid) {
        const int inf = info[key];
        const int body = inf & 0x7fff;
        valid = body > 0 && !(inf & 0x8000);
        bias = valid ? log2f(float(body)) : 0.f;
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

// Key part of an expanded span: c[j][h] = sigma_j g_j (Vt_K q_h)_j * scale*log2(e),
// written to the warp's scratch as [j][8] floats.
__device__ __forceinline__ void consume_expa(WarpAcc& A, const uint8_t* page, int rK,
                                             float* cbuf, float scale_log2) {
  const int lane = threadIdx.x & 31;
  const float* sig = reinterpret_cast<const float*>(page + 16);
  const float* gat = sig + r4(rK);
  const uint32_t vt = smem_u32(page + 16 + 8 * r4(rK));
  for (int nt = 0; nt * 8 < rK; ++nt) {
    float c0 = 0.f, c1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t b0, b1, b2, b3;
      const int row = 8 * nt + (lane & 7);
      ldsm_x4(vt + row * 256 + (32 * i + 8 * (lane >> 3)) * 2, b0, b1, b2, b3);
      mma_bf16_rows8(c0, c1, A.qa[2 * i][0], A.qa[2 * i][1], b0, b1);
      mma_bf16_rows8(c0, c1, A.qa[2 * i + 1][0], A.qa[2 * i + 1][1], b2, b3);
    }
    const int j0 = 8 * nt + 2 * (lane & 3), h = lane >> 2;
    cbuf[j0 * 8 + h] = j0 < rK ? c0 * sig[j0] * gat[j0] * scale_log2 : 0.f;
    cbuf[(j0 + 1) * 8 + h] = (j0 + 1) < rK ? c1 * sig[j0 + 1] * gat[j0 + 1] * scale_log2 : 0.f;
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) A.w[h][0] = A.w[h][1] = 0.f;
  __syncwarp();
}

// U rows of an expanded span: token logits U_K c, online softmax, w += U_V^T p.
__device__ __forceinline__ bool consume_expu(WarpAcc& A, const uint8_t* page, int n, int rK,
                                             int rV, int G, const float* cbuf, float* pbuf) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const __nv_bfloat16* UK = reinterpret_cast<const __nv_bfloat16*>(page);
  const __nv_bfloat16* UV = reinterpret_cast<const __nv_bfloat16*>(page + 16384);
  const float4* c4 = reinterpret_cast<const float4*>(cbuf);
  bool had = false;
  for (int rb = w; rb * 32 < n; rb += kConsumerWarps) {
    had = true;
    const int i = rb * 32 + lane;
    const bool valid = i < n;
    float x[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) x[h] = 0.f;
    if (valid) {
      const __nv_bfloat16* uk = UK + i * rK;
      for (int j = 0; j < rK; ++j) {
        const float u = __bfloat162float(uk[j]);
        const float4 ca = c4[2 * j], cb = c4[2 * j + 1];
        x[0] = fmaf(u, ca.x, x[0]); x[1] = fmaf(u, ca.y, x[1]);
        x[2] = fmaf(u, ca.z, x[2]); x[3] = fmaf(u, ca.w, x[3]);
        x[4] = fmaf(u, cb.x, x[4]); x[5] = fmaf(u, cb.y, x[5]);
        x[6] = fmaf(u, cb.z, x[6]); x[7] = fmaf(u, cb.w, x[7]);
      }
    }
    float my_alpha = 1.f, my_m = A.m_row, my_ps = 0.f;
    const int r0 = lane >> 2;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      if (h < G) {
        const float xv = valid ? x[h] : kNegInf;
        const float mx = warp_max(xv);
        const float m_old = __shfl_sync(0xffffffffu, A.m_row, 4 * h);
        const float m_new = fmaxf(m_old, mx);
        float alpha, msub;
        softmax_rescale(m_old, m_new, alpha, msub);
        const float p = exp2f(xv - msub);
        const float ps = warp_sum(p);
        A.w[h][0] *= alpha;
        A.w[h][1] *= alpha;
        pbuf[lane * 8 + h] = p;
        if (r0 == h) {
          my_alpha = alpha;
          my_m = m_new;
          my_ps = ps;
        }
      } else {
        pbuf[lane * 8 + h] = 0.f;
      }
    }
    A.m_row = my_m;
    A.l_part = fmaf(A.l_part, my_alpha, (lane & 3) == 0 ? my_ps : 0.f);
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      A.o[t][0] *= my_alpha;
      A.o[t][1] *= my_alpha;
    }
    __syncwarp();
    const int nrows = (n - rb * 32) < 32 ? (n - rb * 32) : 32;
    const float4* p4 = reinterpret_cast<const float4*>(pbuf);
    for (int ii = 0; ii < nrows; ++ii) {
      const __nv_bfloat16* uv = UV + (rb * 32 + ii) * rV;
      const float u0 = lane < rV ? __bfloat162float(uv[lane]) : 0.f;
      const float u1 = lane + 32 < rV ? __bfloat162float(uv[lane + 32]) : 0.f;
      const float4 pa = p4[2 * ii], pb = p4[2 * ii + 1];
      const float pp[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        A.w[h][0] = fmaf(pp[h], u0, A.w[h][0]);
        A.w[h][1] = fmaf(pp[h], u1, A.w[h][1]);
      }
    }
    __syncwarp();
  }
  return had;
}

// Value part: o_h += Vt_V^T (sigma_V g_V w_h) for this warp's share of rows.
__device__ __forceinline__ void consume_expb(WarpAcc& A, const uint8_t* page, int rV, int G,
                                             uint8_t* abuf_raw) {
  const int lane = threadIdx.x & 31;
  const float* sig = reinterpret_cast<const float*>(page);
  const float* gat = sig + r4(rV);
  const uint32_t vt = smem_u32(page + 8 * r4(rV));
  // coefficients a[h][j] as bf16 in a 16 x 64 tile, 128B-swizzled rows
  const float s0 = lane < rV ? sig[lane] * gat[lane] : 0.f;
  const float s1 = lane + 32 < rV ? sig[lane + 32] * gat[lane + 32] : 0.f;
  __nv_bfloat16* ab = reinterpret_cast<__nv_bfloat16*>(abuf_raw);
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    const float v0 = (h < 8 && h < G) ? A.w[h & 7][0] * s0 : 0.f;
    const float v1 = (h < 8 && h < G) ? A.w[h & 7][1] * s1 : 0.f;
    const int j0 = lane, j1 = lane + 32;
    ab[(h * 128 + (((j0 >> 3) ^ (h & 7)) << 4) + (j0 & 7) * 2) / 2] = __float2bfloat16_rn(v0);
    ab[(h * 128 + (((j1 >> 3) ^ (h & 7)) << 4) + (j1 & 7) * 2) / 2] = __float2bfloat16_rn(v1);
  }
  __syncwarp();
  const uint32_t abase = smem_u32(abuf_raw);
  const int mi = lane >> 3;
  for (int ks = 0; ks * 16 < rV; ++ks) {
    uint32_t a0, a1, a2, a3;
    const int arow = (lane & 7) + 8 * (mi & 1);
    ldsm_x4(swz128(abase, arow, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
    const int j = 16 * ks + 8 * (mi & 1) + (lane & 7);  // Vt_V row this lane addresses
    const bool tail = 16 * ks + 16 > rV;
    const int jb = 16 * ks + 2 * (lane & 3);             // rows held in b0 / b2 (+8 in b1 / b3)
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vt + j * 256 + (2 * dp + (mi >> 1)) * 16, b0, b1, b2, b3);
      if (tail) {
        const uint32_t lo0 = jb < rV ? 0xffffu : 0u, hi0 = jb + 1 < rV ? 0xffff0000u : 0u;
        const uint32_t lo1 = jb + 8 < rV ? 0xffffu : 0u, hi1 = jb + 9 < rV ? 0xffff0000u : 0u;
        b0 &= lo0 | hi0; b2 &= lo0 | hi0;
        b1 &= lo1 | hi1; b3 &= lo1 | hi1;
      }
      mma_bf16_rows8(A.o[2 * dp][0], A.o[2 * dp][1], a0, a2, b0, b1);
      mma_bf16_rows8(A.o[2 * dp + 1][0], A.o[2 * dp + 1][1], a0, a2, b2, b3);
    }
  }
}

}  // namespace sekv
