// Batched truncated SVD of span bodies (one CTA per body, persistent CTAs).
//
// SeKV, technical summary, Methodik 2 (gist.science, German page) / 方法论 2
// (Chinese page): each span keeps a low-rank SVD basis whose components
// carry soft gates.  For a body M (b x 128, bf16) the kernel forms the Gram
// matrix on the small side (M M^T when b <= 128, else M^T M), diagonalises it
// with the cyclic Jacobi method (Jacobi 1846; rotation formulas as in Golub &
// Van Loan, "Matrix Computations", the symmetric Schur decomposition),
// takes sigma_j = sqrt(lambda_j) in descending order, recovers the other
// factor by projection (v_j = M^T u_j / sigma_j, resp. u_j = M v_j / sigma_j),
// flips each pair so that the largest-magnitude entry of v_j is positive,
// and writes the gated rank-r part into the span's record.
#include "build.cuh"

namespace sekv {

namespace {

__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < int(blockDim.x >> 5); ++w) s += red[w];
  return s;
}

// Circle-method pairing: round r of a tournament among nn (even) players;
// pair k in [0, nn/2).  The pair is left unordered (a Jacobi rotation is
// the same for (p, q) and (q, p)): for k >= 1, p = r + k and q = r - k
// (mod nn - 1) run through consecutive indices as k does, so the threads of
// a warp, one pair each, touch 32 different shared-memory banks.
__device__ __forceinline__ void jacobi_pair(int nn, int r, int k, int& p, int& q) {
  const int m = nn - 1;
  if (k == 0) {
    p = nn - 1;
    q = r;
  } else {
    p = (r + k) % m;
    q = (r - k + m) % m;
  }
}

}  // namespace

template <int NMAX, int NT, bool LARGE>
__global__ void __launch_bounds__(NT) svd_kernel(const BuildParams P, int cls) {
  extern __shared__ __align__(16) uint8_t sm[];
  constexpr int LD = NMAX + 1;
  constexpr int MROWS = LARGE ? 32 : NMAX;                    // body rows staged at once
  float* G = reinterpret_cast<float*>(sm);                    // NMAX x LD
  float* Q = G + NMAX * LD;                                   // NMAX x LD (eigenvectors)
  __nv_bfloat16* Ms = reinterpret_cast<__nv_bfloat16*>(Q + NMAX * LD);  // MROWS x 128
  float* Vs = reinterpret_cast<float*>(Ms + MROWS * kHeadDim);          // LARGE: rank x 128
  float* aux = Vs + (LARGE ? P.rank_cap * kHeadDim : 0);
  float* cs = aux;             // [NMAX/2 + 1]
  float* sn = cs + 72;
  int* pp = reinterpret_cast<int*>(sn + 72);
  int* qq = pp + 72;
  int* ord = qq + 72;          // [NMAX]
  float* red = reinterpret_cast<float*>(ord + 136);  // warp values [32], warp indices [32], sign
  __shared__ int s_item;
  const int tid = threadIdx.x;
  const int count = P.counters[cls];
  const int32_t* list = P.cls_list + size_t(cls) * P.cls_cap;

  for (;;) {
    __syncthreads();
    if (tid == 0) s_item = atomicAdd(&P.counters[4 + cls], 1);
    __syncthreads();
    const int item = s_item;
    if (item >= count || item >= P.cls_cap) break;
    const int code = list[item];
    const int which = code & 1;
    const size_t gk = size_t(code >> 1);
    const int g = int(gk / P.max_spans), k = int(gk % P.max_spans);
    const int b = g / P.Hkv;
    const int bl = P.body_len[size_t(b) * P.max_spans + k];
    const int rank = P.rec_rank[gk];
    const int rK = rank & 0xffff, rV = (rank >> 16) & 0xffff;
    const int r = which ? rV : rK;
    const int t0 = P.starts[size_t(b) * P.max_spans + k] + 1;
    const __nv_bfloat16* M = (which ? P.V : P.K) + (size_t(g) * P.T + t0) * kHeadDim;
    const int n = LARGE ? kHeadDim : bl;
    // records past the store capacity are skipped (plan_kernel flagged them)
    if (P.gbase[g] + P.rel_off[gk] + record_bytes(bl, rK, rV) > P.store_capacity) continue;
    uint8_t* rec = P.store + P.gbase[g] + P.rel_off[gk];

    // ---- Gram matrix on the small side -----------------------------------
    if (!LARGE) {
      const int4* src = reinterpret_cast<const int4*>(M);
      int4* dst = reinterpret_cast<int4*>(Ms);
      for (int i = tid; i < bl * 16; i += NT) dst[i] = src[i];
      __syncthreads();
      for (int e = tid; e < n * n; e += NT) {
        const int i = e / n, j = e % n;
        if (j < i) continue;
        const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(Ms + i * kHeadDim);
        const __nv_bfloat162* c = reinterpret_cast<const __nv_bfloat162*>(Ms + j * kHeadDim);
        // the threads of a warp hold different j: starting each row at pair
        // (d + j) mod 64 spreads their reads of rows j over the banks (rows
        // 256 bytes apart all start in bank 0)
        float acc = 0.f;
#pragma unroll 8
        for (int d = 0; d < kHeadDim / 2; ++d) {
          const float2 x = __bfloat1622float2(a[(d + j) & 63]);
          const float2 y = __bfloat1622float2(c[(d + j) & 63]);
          acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
        }
        G[i * LD + j] = acc;
        G[j * LD + i] = acc;
      }
    } else {
      // M^T M (128 x 128), rows streamed through Ms in chunks of NMAX rows
      constexpr int PAIRS = (kHeadDim * (kHeadDim + 1) / 2 + NT - 1) / NT;
      float acc[PAIRS];
      int pi[PAIRS], pj[PAIRS];
#pragma unroll
      for (int t = 0; t < PAIRS; ++t) {
        acc[t] = 0.f;
        int e = tid + t * NT, i = 0;
        // map e to (i, j) with i <= j in the upper triangle, row-major
        while (e >= kHeadDim - i && i < kHeadDim) {
          e -= kHeadDim - i;
          ++i;
        }
        pi[t] = i;
        pj[t] = i + e;
      }
      for (int r0 = 0; r0 < bl; r0 += MROWS) {
        const int rows = min(MROWS, bl - r0);
        __syncthreads();
        const int4* src = reinterpret_cast<const int4*>(M + size_t(r0) * kHeadDim);
        int4* dst = reinterpret_cast<int4*>(Ms);
        for (int i = tid; i < rows * 16; i += NT) dst[i] = src[i];
        __syncthreads();
        for (int rr = 0; rr < rows; ++rr) {
          const __nv_bfloat16* row = Ms + rr * kHeadDim;
#pragma unroll
          for (int t = 0; t < PAIRS; ++t)
            if (pi[t] < kHeadDim)
              acc[t] = fmaf(__bfloat162float(row[pi[t]]), __bfloat162float(row[pj[t]]), acc[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < PAIRS; ++t)
        if (pi[t] < kHeadDim) {
          G[pi[t] * LD + pj[t]] = acc[t];
          G[pj[t] * LD + pi[t]] = acc[t];
        }
    }
    // Q = I; an odd n pairs its last index with a dummy index n in every
    // round of the tournament, whose row and column of G and column of Q are
    // kept zero (its rotation is the identity)
    constexpr int NX = NMAX / 2 < 32 ? NMAX / 2 : 32;  // pair (column) lanes
    constexpr int NY = NT / NX;                        // row lanes
    constexpr int BPT = (NMAX / 2 + NX - 1) / NX;      // column pairs per thread
    const int tx = tid % NX, ty = tid / NX;
    const int nn = (n + 1) & ~1, np = nn / 2;
    for (int i = ty; i < nn; i += NY)
      for (int j = tx; j < nn; j += NX) {
        Q[i * LD + j] = (i == j && i < n) ? 1.f : 0.f;
        if (i >= n || j >= n) G[i * LD + j] = 0.f;
      }
    __syncthreads();

    // ---- cyclic Jacobi, parallel (tournament) ordering ---------------------
    // One round rotates nn/2 disjoint pairs at once: G <- J^T G J and Q <- Q J
    // with J the product of the round's rotations.  Each 2x2 block of G
    // (rows of pair a, columns of pair b) is updated in one step,
    // R_a^T G_ab R_b, so a round needs one barrier after the rotations and one
    // after the update.
    int sweeps = 0;  // sweeps that rotated (for the operation count)
    for (int sweep = 0; sweep < 24; ++sweep) {
      float off = 0.f, dg = 0.f;
      for (int i = ty; i < n; i += NY)
        for (int j = tx; j < n; j += NX) {
          const float v = G[i * LD + j];
          if (i == j) dg += v * v; else off += v * v;
        }
      off = block_sum(off, red);
      dg = block_sum(dg, red);
      // fp32 rotations leave off-diagonal energy near 1e-13 of the diagonal's;
      // stop once it is under 1e-12 of it (inside the build's accuracy bars:
      // sigma 1e-3 relative, reconstruction 5e-3)
      if (!(off > 1e-12f * dg)) break;
      ++sweeps;
      for (int rd = 0; rd < nn - 1; ++rd) {
        if (tid < np) {
          int p, q;
          jacobi_pair(nn, rd, tid, p, q);
          float c = 1.f, s = 0.f;
          if (p < n && q < n) {
            const float apq = G[p * LD + q];
            if (apq != 0.f) {
              // tan of the rotation angle, smaller root (Golub & Van Loan);
              // rsqrt keeps c^2 + s^2 = 1 to a few ulp, which is all the
              // orthogonality of Q needs
              const float theta = __fdividef(G[q * LD + q] - G[p * LD + p], 2.f * apq);
              float t;
              if (fabsf(theta) > 1e18f) {
                t = __fdividef(0.5f, theta);
              } else {
                const float u = fmaf(theta, theta, 1.f);
                t = __fdividef(1.f, fabsf(theta) + u * rsqrtf(u));
                if (theta < 0.f) t = -t;
              }
              c = rsqrtf(fmaf(t, t, 1.f));
              s = t * c;
            }
          }
          cs[tid] = c;
          sn[tid] = s;
          pp[tid] = p;
          qq[tid] = q;
        }
        __syncthreads();
        int pb[BPT], qb[BPT];
        float cb[BPT], sb[BPT];
#pragma unroll
        for (int t = 0; t < BPT; ++t) {
          const int b = tx + t * NX;
          const bool ok = b < np;
          pb[t] = ok ? pp[b] : 0;
          qb[t] = ok ? qq[b] : 0;
          cb[t] = ok ? cs[b] : 1.f;
          sb[t] = ok ? sn[b] : 0.f;
        }
        for (int a = ty; a < np; a += NY) {
          const int pa = pp[a], qa = qq[a];
          const float ca = cs[a], sa = sn[a];
#pragma unroll
          for (int t = 0; t < BPT; ++t) {
            if (tx + t * NX >= np) break;
            float* gp = G + pa * LD;
            float* gq = G + qa * LD;
            const float x = gp[pb[t]], y = gp[qb[t]], z = gq[pb[t]], w = gq[qb[t]];
            const float x1 = ca * x - sa * z, y1 = ca * y - sa * w;
            const float z1 = sa * x + ca * z, w1 = sa * y + ca * w;
            gp[pb[t]] = cb[t] * x1 - sb[t] * y1;
            gp[qb[t]] = sb[t] * x1 + cb[t] * y1;
            gq[pb[t]] = cb[t] * z1 - sb[t] * w1;
            gq[qb[t]] = sb[t] * z1 + cb[t] * w1;
          }
        }
        for (int i = ty; i < n; i += NY) {
          float* qi = Q + i * LD;
#pragma unroll
          for (int t = 0; t < BPT; ++t) {
            if (tx + t * NX >= np) break;
            const float vp = qi[pb[t]], vq = qi[qb[t]];
            qi[pb[t]] = cb[t] * vp - sb[t] * vq;
            qi[qb[t]] = sb[t] * vp + cb[t] * vq;
          }
        }
        __syncthreads();
      }
    }
    __syncthreads();
    if (tid == 0 && P.flops != nullptr) {
      // fp32 operations of this body (an fma counts 2): the Gram matrix, every
      // sweep's norms and rotations of G's rows and columns and of the
      // eigenvectors (3 per element and rotation), and the projection onto
      // the other side for the r kept components
      const unsigned long long nq = (unsigned long long)n;
      const unsigned long long gram =
          LARGE ? 128ull * 129ull * (unsigned long long)bl : nq * (nq + 1ull) * 128ull;
      const unsigned long long sweep_ops =
          2ull * nq * nq + (unsigned long long)(nn - 1) * (nn / 2) * nq * 18ull;
      const unsigned long long proj = 2ull * (unsigned long long)r * 128ull * (unsigned long long)bl;
      atomicAdd(P.flops, gram + (unsigned long long)sweeps * sweep_ops + proj);
    }
    // ---- order eigenvalues descending (ties by index) ----------------------
    for (int i = tid; i < n; i += NT) {
      const float li = G[i * LD + i];
      int rk = 0;
      for (int m = 0; m < n; ++m) {
        const float lm = G[m * LD + m];
        rk += (lm > li) || (lm == li && m < i);
      }
      ord[rk] = i;
    }
    __syncthreads();

    // ---- factors, signs, record -------------------------------------------
    const int r4v = r4(r), rs = r8(r);  // U rows hold r8(r) columns, the last ones zero
    const RecordLayout RL = record_layout(bl, rK, rV);
    uint8_t* part;       // sigma/g/Vt of this side
    __nv_bfloat16* Ud;   // U of this side
    if (which == 0) {
      if (tid == 0) {
        int4* h = reinterpret_cast<int4*>(rec);
        *h = make_int4(bl, rK, rV, 0);
        P.rec_off[gk] = P.gbase[g] + P.rel_off[gk];
      }
      part = rec + 16;
      Ud = reinterpret_cast<__nv_bfloat16*>(rec + RL.uk);
    } else {
      part = rec + RL.vpart;
      Ud = reinterpret_cast<__nv_bfloat16*>(rec + RL.uv);
    }
    float* sig = reinterpret_cast<float*>(part);
    float* gat = sig + r4v;
    __nv_bfloat16* Vt = reinterpret_cast<__nv_bfloat16*>(part + 8 * r4v);
    const float* gin = P.gates + ((size_t(b) * P.Hkv + (g % P.Hkv)) * 2 * P.max_spans +
                                  size_t(which) * P.max_spans + k) * P.rank_cap;
    for (int j = tid; j < r4v; j += NT) {
      const float lam = j < r ? G[ord[j] * LD + ord[j]] : 0.f;
      sig[j] = j < r ? sqrtf(fmaxf(lam, 0.f)) : 0.f;
      gat[j] = j < r ? gin[j] : 0.f;
    }
    for (int e = tid; e < bl * (rs - r); e += NT)  // zero padding columns of U
      Ud[size_t(e / (rs - r)) * rs + u_col(e / (rs - r), r + e % (rs - r), rs)] =
          __float2bfloat16_rn(0.f);
    for (int j = 0; j < r; ++j) {
      const int col = ord[j];
      const float sj = sqrtf(fmaxf(G[col * LD + col], 0.f));
      const float inv = sj > 1e-30f ? 1.f / sj : 0.f;
      // v_j (128 dims): projection (small side) or the eigenvector (large side)
      float v[(kHeadDim + NT - 1) / NT];
      float best = -1.f;
      int bidx = kHeadDim;
#pragma unroll
      for (int t = 0; t < (kHeadDim + NT - 1) / NT; ++t) {
        const int d = tid + t * NT;
        float x = 0.f;
        if (d < kHeadDim) {
          if (!LARGE) {
            for (int i = 0; i < bl; ++i)
              x = fmaf(Q[i * LD + col], __bfloat162float(Ms[i * kHeadDim + d]), x);
            x *= inv;
          } else {
            x = sj > 1e-30f ? Q[d * LD + col] : 0.f;
          }
          if (fabsf(x) > best || (fabsf(x) == best && d < bidx)) {
            best = fabsf(x);
            bidx = d;
          }
        }
        v[t] = x;
      }
      // arg max |v_j| over the block (lowest index on ties)
      {
        const int lane = tid & 31, wid = tid >> 5;
        for (int o = 16; o; o >>= 1) {
          const float ob = __shfl_xor_sync(0xffffffffu, best, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
          if (ob > best || (ob == best && oi < bidx)) {
            best = ob;
            bidx = oi;
          }
        }
        __syncthreads();
        if (lane == 0) {
          red[wid] = best;
          reinterpret_cast<int*>(red)[32 + wid] = bidx;
        }
        __syncthreads();
        best = red[0];
        bidx = reinterpret_cast<int*>(red)[32];
        for (int w = 1; w < NT / 32; ++w) {
          const float ob = red[w];
          const int oi = reinterpret_cast<int*>(red)[32 + w];
          if (ob > best || (ob == best && oi < bidx)) {
            best = ob;
            bidx = oi;
          }
        }
      }
      // sign of the winning entry: recompute it from the owner's value
      __syncthreads();
#pragma unroll
      for (int t = 0; t < (kHeadDim + NT - 1) / NT; ++t)
        if (tid + t * NT == bidx) red[64] = v[t];
      __syncthreads();
      const float sgn = red[64] < 0.f ? -1.f : 1.f;
#pragma unroll
      for (int t = 0; t < (kHeadDim + NT - 1) / NT; ++t) {
        const int d = tid + t * NT;
        if (d < kHeadDim) {
          // rows are stored with their 16-byte chunks swizzled by (row & 7)
          Vt[j * kHeadDim + ((((d >> 3) ^ (j & 7)) << 3) | (d & 7))] = __float2bfloat16_rn(sgn * v[t]);
          if (LARGE) Vs[j * kHeadDim + d] = sgn * v[t];
        }
      }
      if (!LARGE) {
        for (int i = tid; i < bl; i += NT)
          Ud[size_t(i) * rs + u_col(i, j, rs)] = __float2bfloat16_rn(sgn * Q[i * LD + col]);
      }
    }
    if (LARGE && r > 0) {
      // u_j = M v_j / sigma_j, rows streamed through Ms
      __syncthreads();
      for (int r0 = 0; r0 < bl; r0 += MROWS) {
        const int rows = min(MROWS, bl - r0);
        __syncthreads();
        const int4* src = reinterpret_cast<const int4*>(M + size_t(r0) * kHeadDim);
        int4* dst = reinterpret_cast<int4*>(Ms);
        for (int i = tid; i < rows * 16; i += NT) dst[i] = src[i];
        __syncthreads();
        for (int e = tid; e < rows * r; e += NT) {
          const int i = e / r, j = e % r;
          const int col = ord[j];
          const float sj = sqrtf(fmaxf(G[col * LD + col], 0.f));
          float acc = 0.f;
          for (int d = 0; d < kHeadDim; ++d)
            acc = fmaf(__bfloat162float(Ms[i * kHeadDim + d]), Vs[j * kHeadDim + d], acc);
          Ud[size_t(r0 + i) * rs + u_col(r0 + i, j, rs)] =
              __float2bfloat16_rn(sj > 1e-30f ? acc / sj : 0.f);
        }
      }
    }
  }
}

namespace {
template <int NMAX, int NT, bool LARGE>
cudaError_t launch_svd(const BuildParams& P, int cls, int sms, cudaStream_t stream) {
  const int smem = svd_smem_bytes(NMAX, LARGE, P.rank_cap);
  auto kern = svd_kernel<NMAX, NT, LARGE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  kern<<<sms * per_sm, NT, smem, stream>>>(P, cls);
  return cudaGetLastError();
}
}  // namespace

// One persistent launch per size class (the class lists come from plan_kernel).
cudaError_t launch_svd_all(const BuildParams& P, int sms, cudaStream_t stream) {
  cudaError_t e = launch_svd<32, 64, false>(P, 0, sms, stream);
  if (e == cudaSuccess) e = launch_svd<64, 256, false>(P, 1, sms, stream);
  if (e == cudaSuccess) e = launch_svd<128, 1024, false>(P, 2, sms, stream);
  if (e == cudaSuccess) e = launch_svd<128, 512, true>(P, 3, sms, stream);
  return e;
}

}  // namespace sekv
