// Parameters of the routing and fetch kernels (shared by host and device).
#pragma once

#include "sekv_common.cuh"

namespace sekv {

constexpr int kRouteChunk = 256;   // spans per routing CTA (one per thread)
constexpr int kRouteThreads = 256;
constexpr int kRouteMaxChunks = 1024;  // max_spans <= 262144

struct RouteParams {
  const int32_t* n_spans;
  const int32_t* body_len;
  const float* s_route;
  const __nv_bfloat16* q;
  const float* W_r;
  const float* theta;
  int32_t* expanded;
  int32_t* n_expanded;
  float* z_out;
  int32_t* status;
  GroupState* groups;
  int32_t* list_scratch;  // [B*Hkv][max_spans]
  int32_t* cnt_scratch;   // [B*Hkv][chunks]
  int B, Hq, Hkv, G, max_spans, chunks;
};

constexpr int kFetchParts = 48;
constexpr int kFetchUnroll = 8;  // 16-byte loads in flight per thread

struct FetchParams {
  const int32_t* n_spans;
  const int32_t* body_len;
  const int64_t* rec_off;
  const int32_t* rec_rank;
  const uint8_t* store;  // device-addressable host memory
  const int32_t* expanded;
  const int32_t* n_expanded;
  uint8_t* staging;
  int64_t per_group;
  int64_t* staged_off;
  int32_t* status;
  int Hkv, max_spans;
};

__global__ void route_kernel(const RouteParams P);
__global__ void fetch_kernel(const FetchParams P);

}  // namespace sekv
