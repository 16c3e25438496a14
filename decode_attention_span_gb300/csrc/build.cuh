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
  // decode-time maintenance: summaries of spans only_k[b] .. only_k[b] +
  // only_n[b] - 1 of each sequence instead of every span; null in the
  // prefill build
  const int32_t* only_k;
  const int32_t* only_n;
  int B, Hkv, T, n_sink, n_recent, max_spans, rank_cap, len_min, len_max;
  float tau;
};

// Decode-time maintenance of one layer's cache (sekv_append_token): the new
// token joins the tail of the full-resolution rows; the token leaving the
// recent window continues the segmentation walk; a span it closes is built by
// the build's summary and SVD kernels (run in place on the full rows: K = the
// full rows of each group, T = their capacity, H = the tail surprisal by row).
struct MaintParams {
  const __nv_bfloat16* k_new;  // [B][Hkv][128]
  const __nv_bfloat16* v_new;
  const float* h_new;          // [B]
  const float* gates;          // [B][Hkv][2][max_spans][rank_cap]
  int32_t* n_spans;
  int32_t* n_tail;
  int32_t* body_len;
  __nv_bfloat16* k_full;
  __nv_bfloat16* v_full;
  float* s_route;
  __nv_bfloat16* k_sum;
  __nv_bfloat16* v_sum;
  int64_t* rec_off;
  int32_t* rec_rank;
  int64_t store_capacity;
  // maintenance state (caller-owned, kept across calls)
  int32_t* seq_len;                // [B] sequence lengths
  int32_t* s_open;                 // [B] the open span's anchor position, -1: none
  int32_t* n_pend;                 // [B] closed spans not yet built (head of the tail)
  int32_t* pend_rows;              // [B] their rows (anchors and bodies)
  int32_t* pend_len;               // [B][kMaxPending] their lengths, in order
  unsigned long long* store_used;  // bytes of the store in use (records go after)
  int32_t* pend;                   // [B][8] init: the values to commit
  int32_t* only_k;                 // [B] first ordinal a flush builds
  int32_t* only_n;                 // [B] how many it builds
  float* tail_h;                   // [B][cap] surprisal of the token in each full row
  // build workspace
  int32_t* status;
  int32_t* starts;
  int64_t* rel_off;
  int64_t* gbase;
  int32_t* counters;
  int32_t* cls_list;
  int64_t cls_cap;
  int B, Hkv, T, cap, n_sink, n_recent, max_spans, rank_cap, len_min, len_max;  // T: init only
  float tau;
};

__global__ void maint_init_rows_kernel(const MaintParams M, const __nv_bfloat16* K,
                                       const __nv_bfloat16* V, const float* H);
__global__ void maint_init_commit_kernel(const MaintParams M);
__global__ void maint_used_kernel(const MaintParams M);
__global__ void maint_append_kernel(const MaintParams M);
__global__ void maint_flush_plan_kernel(const MaintParams M);
__global__ void maint_flush_move_kernel(const MaintParams M);
__global__ void maint_flush_commit_kernel(const MaintParams M);

// closed spans a sequence can hold unbuilt (a flush is needed before more)
constexpr int kMaxPending = 128;

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
