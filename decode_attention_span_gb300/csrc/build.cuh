// Prefill build of one layer's span cache: shared parameters.
//
// SeKV, technical summary (gist.science, German page / Chinese page):
// Methodik 1 / 方法论 1 (surprisal-threshold segmentation, anchors),
// Methodik 2 / 方法论 2 (routing summary: normalised surprisal-weighted mean
// of projected keys; per-span low-rank SVD basis with soft rank gates).
#pragma once

#include "sekv_common.cuh"

namespace sekv {

// SVD work classes by the small side of the span body (b x 128):
//   0: b <= 32, 1: b <= 64, 2: b <= 128 (Gram M M^T), 3: b > 128 (Gram M^T M)
constexpr int kSvdClasses = 4;

struct BuildParams {
  // inputs
  const __nv_bfloat16* K;  // [B][Hkv][T][128]
  const __nv_bfloat16* V;
  const float* H;          // [B][T]
  const float* W_r;        // [Hkv][64][128]
  const float* gates;      // [B][Hkv][2][max_spans][rank_cap]
  // outputs (one layer of the cache)
  int32_t* n_spans;
  int32_t* body_len;
  __nv_bfloat16* k_full;
  __nv_bfloat16* v_full;
  float* s_route;
  __nv_bfloat16* k_sum;
  __nv_bfloat16* v_sum;
  int64_t* rec_off;
  int32_t* rec_rank;
  uint8_t* store;
  int64_t store_capacity;
  // workspace
  int32_t* status;
  unsigned long long* flops;  // fp32 operations the span SVDs performed (fma = 2), summed
  int32_t* starts;         // [B][max_spans] anchor positions
  int64_t* rel_off;        // [B*Hkv][max_spans] record offset within its group
  int64_t* gtotal;         // [B*Hkv]
  int64_t* gbase;          // [B*Hkv]
  int32_t* counters;       // [0..3] class counts, [4..7] class cursors, [8] plan CTAs done
  int32_t* cls_list;       // [4][B*Hkv*max_spans*2]
  int64_t cls_cap;
  int B, Hkv, T, n_sink, n_recent, max_spans, rank_cap, len_min, len_max;
  float tau;
};

__global__ void seg_kernel(const BuildParams P);
__global__ void plan_kernel(const BuildParams P);
__global__ void gather_kernel(const BuildParams P);
__global__ void summary_kernel(const BuildParams P);
cudaError_t launch_svd_all(const BuildParams& P, int sms, cudaStream_t stream);

// shared memory bytes of one svd_kernel CTA
__host__ __device__ constexpr int svd_smem_bytes(int nmax, bool large, int rcap) {
  return 2 * nmax * (nmax + 1) * 4 + (large ? 32 : nmax) * 256 + (large ? rcap * 128 * 4 : 0) +
         4096;
}

}  // namespace sekv
