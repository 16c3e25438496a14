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
constexpr int kFetchUnroll = 16;  // 16-byte loads in flight per thread

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

// Residency cache of basis records (sekv_fetch_bases_cached): the table's
// arrays, the copy plan in the workspace, and the pool's place in staging.
struct CacheParams {
  const int32_t* n_spans;
  const int32_t* body_len;
  const int64_t* rec_off;
  const int32_t* rec_rank;
  const uint8_t* store;     // device-addressable host memory
  const int32_t* expanded;
  const int32_t* n_expanded;
  uint8_t* staging;
  int64_t per_group;
  int64_t pool_base;        // byte offset of the slots in staging (B*Hkv*per_group)
  int32_t* slot_of;         // [g][max_spans]
  int32_t* span_of;         // [g][n_slots]
  int32_t* stamp;           // [g][n_slots]
  int32_t* epoch;           // [g]
  int32_t* hand;            // [g]
  int64_t* plan;            // [g][max_spans][3]: source offset, staging offset, bytes
  int32_t* plan_n;          // [g]
  int64_t* staged_off;
  int32_t* hits;            // [g] or null
  int64_t* copied;          // [g] or null: record bytes copied
  int32_t* status;
  int Hkv, max_spans, n_slots, slot_bytes;
};

constexpr int kCacheMaxSlots = 4096;  // slots per group (the plan kernel's shared list)

__global__ void route_kernel(const RouteParams P);
__global__ void fetch_kernel(const FetchParams P);
__global__ void cache_plan_kernel(const CacheParams P);
__global__ void cache_copy_kernel(const CacheParams P);

}  // namespace sekv
