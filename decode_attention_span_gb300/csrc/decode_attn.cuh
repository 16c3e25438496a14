// Mixed-resolution decode attention over the span cache (one layer).
//
// SeKV, technical summary, Methodik 3 (gist.science, German page) / 方法论 3
// (Chinese page): the query is routed against the span summaries; sink,
// anchor and recent rows enter the attention at full resolution,
// unexpanded spans enter once with their summary key/value and the size
// correction ln|S|, expanded spans enter with their token-level keys/values
// rebuilt from the gated low-rank basis.  This kernel scores expanded spans
// in factor space: c = diag(sigma g) Vt_K q, logits = U_K c; then
// w = U_V^T p and o += Vt_V^T diag(sigma g) w; khat/vhat are never formed.
//
// Structure (one CTA per (sequence, KV head, chunk); 1 CTA per SM):
//   warp 4 (producer): streams fixed-size pages into a 4-slot shared-memory
//     ring with TMA (3-D tiled copies, 128B swizzle, for full-resolution
//     rows, summary rows and routing summaries; 1-D bulk copies for basis
//     records), tracked by full/empty mbarriers.
//   warps 0-3 (consumers): route (fused mode), then run an online softmax
//     over the pages with mma.sync (query heads of the GQA group as the M
//     rows, keys as N), FMA for the U factors.
//   Split-KV: every CTA owns an equal share of the fixed bytes (routing
//     summaries, full rows, summary rows); the expanded spans of a KV head
//     are shared out by bytes once all its CTAs have published what they
//     expand; the last CTA of a KV head merges the partial softmax states.
#pragma once

#include "sekv_common.cuh"

namespace sekv {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kPages = 4;
constexpr int kPageData = 32768;
constexpr int kPageStride = 34816;  // 32 KB data + 2 KB aux, 1024-aligned
constexpr int kAuxBody = 32768;
constexpr int kAuxRank = 33280;
constexpr int kAuxOff = 33792;
constexpr int kScratchPerWarp = 3072;
constexpr int kInfoCap = 2048;       // span-info cache entries per CTA
constexpr int kRouteSpans = 128;     // spans per routing page
constexpr int kTileRows = 64;        // rows per full/summary page
constexpr int kMaxCgSmem = 256;      // CTAs per KV head the producer can index

constexpr int kMaxRecPerPage = 8;   // small basis records packed into one page
constexpr int kWrStride = 528;      // W_r rows in shared memory (512 B + 16 B pad)

constexpr int kOffScratch = kPages * kPageStride;
constexpr int kOffInfo = kOffScratch + kConsumerWarps * kScratchPerWarp;
constexpr int kOffWr = kOffInfo + kInfoCap * 4;   // info cache: one float per span
constexpr int kOffMisc = kOffWr + kRouteDim * kWrStride;
constexpr int kMiscBytes = 4608;
constexpr int kSmemBytes = kOffMisc + kMiscBytes;
constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment

enum PageType : int {
  PG_ROUTE = 1, PG_INFO = 2, PG_FULL = 3, PG_SUM = 4, PG_EXP = 5, PG_END = 6, PG_EXPM = 7
};

// One basis record inside a PG_EXPM page (several small records per page).
struct RecInfo {
  int off;  // byte offset in the page
  int b, rk, rv;
};

struct PageDesc {
  int type;
  int n;       // rows / spans / body tokens in this page
  int a;       // first row / first span ordinal / first body token
  int rk, rv;  // expanded span: ranks
  int flag;    // ROUTE: last routing page
  int off_a;   // EXP: byte offset of the key part (header..Vt_K) or -1
  int off_uk;  // EXP: byte offset of U_K rows [a, a+n)
  int off_uv;  // EXP: byte offset of U_V rows [a, a+n)
  int off_b;   // EXP: byte offset of the value part (sigma_V..Vt_V) or -1
  int pad0, pad1;
};

struct DecodeParams {
  CUtensorMap tm_kfull, tm_vfull, tm_ksum, tm_vsum, tm_sroute;
  const int32_t* n_spans;
  const int32_t* body_len;
  const int64_t* rec_off;
  const int32_t* rec_rank;
  const uint8_t* store;  // base that entry offsets refer to (store or staging)
  const __nv_bfloat16* q;
  const float* W_r;
  const float* theta;
  float* out;
  float* lse;
  int32_t* expanded_out;
  int32_t* n_expanded_out;
  int32_t* status;
  GroupState* groups;
  int32_t* cta_n;
  int64_t* cta_bytes;
  ExpEntry* entries;
  const uint16_t* info;  // list mode: per-span info written by the prep kernel
  Partial* partials;
  int B, Hq, Hkv, G, n_sink, n_recent, max_spans, cap_full, cg;
  float scale_log2;
  int fused;
};

struct PrepParams {
  const int32_t* n_spans;
  const int32_t* body_len;
  const int64_t* rec_off;
  const int32_t* rec_rank;
  const int32_t* expanded;
  const int32_t* n_expanded;
  const int64_t* staged_off;
  int32_t* status;
  GroupState* groups;
  int32_t* cta_n;
  int64_t* cta_bytes;
  ExpEntry* entries;
  uint16_t* info;
  int Hkv, max_spans, cg;
};

__global__ void decode_kernel(const __grid_constant__ DecodeParams P);
__global__ void prep_list_kernel(const PrepParams P);

// Fixed-part split: rows cost 2 units (512 B of K+V), spans 3 units in fused
// mode (512 B of summary K+V plus 256 B of routing summary) or 2 in list mode.
// Span boundaries are rounded up to multiples of 8 so that every per-span
// array slice starts 16-byte aligned.
__host__ __device__ inline void fixed_range(int j, int cg, int n_full, int n_sp, int fused,
                                            int& f0, int& f1, int& k0, int& k1) {
  const int64_t ws = fused ? 3 : 2;
  const int64_t U = 2 * int64_t(n_full) + ws * int64_t(n_sp);
  const int64_t x0 = U * j / cg, x1 = U * (j + 1) / cg;
  auto fpos = [&](int64_t x) -> int {
    int64_t v = (x + 1) / 2;
    return int(v < n_full ? v : n_full);
  };
  auto kpos = [&](int64_t x) -> int {
    int64_t r = x - 2 * int64_t(n_full);
    if (r <= 0) return 0;
    int64_t v = (r + ws - 1) / ws;
    v = (v + 7) & ~int64_t(7);
    return int(v < n_sp ? v : n_sp);
  };
  f0 = fpos(x0);
  f1 = fpos(x1);
  k0 = kpos(x0);
  k1 = kpos(x1);
}

struct SmemMisc {
  PageDesc desc[kPages];
  RecInfo rec[kPages][kMaxRecPerPage];
  uint64_t full[kPages];
  uint64_t empty[kPages];
  uint64_t wr_bar;   // W_r rows staged in shared memory (fused mode)
  int n_local;
  int wcnt[kConsumerWarps];
  int is_last;
  int abort_flag;
  int pad0;
  long long bytes_local;
  long long wbytes[kConsumerWarps];
  float theta[8];
  int pre_n[kMaxCgSmem + 1];
  long long pre_b[kMaxCgSmem + 1];
};
static_assert(sizeof(SmemMisc) <= kMiscBytes, "misc smem");

constexpr uint32_t kWaitLimit = 1u << 24;  // bounded mbarrier polls (~1-2 s at most)
constexpr uint32_t kSpinLimit = 1u << 22;  // bounded polls of global counters (~2-3 s)

// ----------------------------------------------------------------------------
// producer (one lane issues; the whole warp helps in the expanded phase)
// ----------------------------------------------------------------------------
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
};

__device__ __forceinline__ uint8_t* page_ptr(uint8_t* smem, int slot) {
  return smem + slot * kPageStride;
}

// Wait for a free slot, publish the descriptor (and the record table of a
// multi-record page) and only then arm the full barrier, so that the
// consumers' acquire on the barrier covers both.
__device__ __forceinline__ uint8_t* push_page(uint8_t* smem, SmemMisc* ms, Ring& r,
                                              const PageDesc& d, uint32_t bytes,
                                              int32_t* status, bool& ok,
                                              const RecInfo* tab = nullptr, int ntab = 0) {
  if (!mbar_wait(&ms->empty[r.slot], r.phase ^ 1u, kWaitLimit)) {
    set_device_error(status, DEV_WAIT_TIMEOUT, 1);
    ok = false;
    return nullptr;
  }
  ms->desc[r.slot] = d;
  for (int i = 0; i < ntab; ++i) ms->rec[r.slot][i] = tab[i];
  mbar_arrive_expect_tx(&ms->full[r.slot], bytes);
  return page_ptr(smem, r.slot);
}

__device__ __forceinline__ void advance(Ring& r) {
  if (++r.slot == kPages) {
    r.slot = 0;
    r.phase ^= 1u;
  }
}

}  // namespace sekv
