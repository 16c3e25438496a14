// List preparation kernel of sekv_decode_attention (span info and the
// expansion entries from a caller's ascending list).
#include "decode_attn.cuh"

namespace sekv {

// ----------------------------------------------------------------------------
// list mode: span info and expansion entries from a caller's ascending list
// ----------------------------------------------------------------------------


__global__ void __launch_bounds__(256) prep_list_kernel(const PrepParams P) {
  __shared__ long long scan[256];
  __shared__ long long carry;
  const int g = blockIdx.x, b = g / P.Hkv, tid = threadIdx.x;
  const size_t gs = size_t(g) * P.max_spans;
  const int n_sp = P.n_spans[b];
  int ne = P.n_expanded[g];
  if (ne < 0 || ne > n_sp) {
    if (tid == 0) set_device_error(P.status, DEV_BAD_LIST, g);
    ne = 0;
  }
  for (int k = tid; k < n_sp; k += 256)
    P.info[gs + k] = uint16_t(P.body_len[size_t(b) * P.max_spans + k] & 0x7fff);
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int e0 = 0; e0 < ne; e0 += 256) {
    const int e = e0 + tid;
    long long size = 0;
    int k = -1, body = 0, rank = 0;
    if (e < ne) {
      k = P.expanded[gs + e];
      const int prev = e > 0 ? P.expanded[gs + e - 1] : -1;
      bool okk = k >= 0 && k < n_sp && k > prev;
      if (okk) {
        body = P.body_len[size_t(b) * P.max_spans + k];
        rank = P.rec_rank[gs + k];
        okk = body > 0 && (rank & 0xffff) <= SEKV_MAX_RANK && ((rank >> 16) & 0xffff) <= SEKV_MAX_RANK;
      }
      if (!okk) {
        set_device_error(P.status, DEV_BAD_LIST, e);
        body = 0;
      } else {
        size = record_bytes(body, rank & 0xffff, (rank >> 16) & 0xffff);
      }
    }
    scan[tid] = size;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {
      const long long v = tid >= o ? scan[tid - o] : 0;
      __syncthreads();
      scan[tid] += v;
      __syncthreads();
    }
    const long long cum = carry + scan[tid] - size;
    if (e < ne) {
      const long long off = body > 0 ? (P.staged_off ? P.staged_off[gs + e] : P.rec_off[gs + k]) : 0;
      int4* dst = reinterpret_cast<int4*>(P.entries + gs + e);
      dst[0] = make_int4(k, body, rank, 0);
      dst[1] = make_int4(int(uint32_t(off)), int(off >> 32), int(uint32_t(cum)), int(cum >> 32));
      if (body > 0) P.info[gs + k] = uint16_t((body & 0x7fff) | 0x8000);
    }
    __syncthreads();
    if (tid == 255) carry += scan[255];
    __syncthreads();
  }
  for (int jj = tid; jj < P.cg; jj += 256) {
    P.cta_n[size_t(g) * P.cg + jj] = jj == 0 ? ne : 0;
    P.cta_bytes[size_t(g) * P.cg + jj] = jj == 0 ? carry : 0;
  }
  if (tid == 0) P.groups[g].published = P.cg;
}

}  // namespace sekv
