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
// Structure (one CTA per (sequence, KV head, chunk); one CTA per SM):
//   warp 4 (producer): streams pages into per-warp rings (two 19 KB slots per
//     consumer warp) with TMA: 3-D tiled copies with 128B swizzle for
//     full-resolution rows, summary rows, routing summaries and W_r; 1-D
//     bulk copies for basis records.  Full/empty mbarriers per slot.
//   warps 0-3 (consumers): each consumes its own ring independently and keeps
//     its own online-softmax state (query heads of the GQA group as the M rows
//     of mma.sync; keys, tokens or ranks as N).  The four states and then the
//     CTAs' partial states are merged at the end.
//   Work split: every CTA owns an equal share of the fixed bytes (routing
//     summaries, full rows, summary rows), dealt to its warps round-robin; the
//     expanded spans of a KV head are shared out among its CTAs by bytes once
//     all of them have published what they expand, and inside a CTA each
//     record goes to the least-loaded warp.
#pragma once

#include "sekv_common.cuh"

namespace sekv {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kSlotsPerWarp = 2;
constexpr int kSlots = kConsumerWarps * kSlotsPerWarp;
constexpr int kSlotBytes = 19456;     // 18 KB of data, 1024-aligned (19 KB)
constexpr int kPageData = 18432;      // bytes of data a page may hold
constexpr int kTileRows = 32;         // rows per full / summary page
constexpr int kBoxBytes = kTileRows * 128;  // one 128B-swizzled box: 32 rows x 64 bf16
constexpr int kRouteSpans = 64;       // spans per routing page
constexpr int kInfoCap = 2048;        // span-info cache entries per CTA
constexpr int kMaxRoutePages = kInfoCap / kRouteSpans;
constexpr int kMaxCgSmem = 256;       // CTAs per KV head the producer can index
constexpr int kMaxRecPerPage = 8;     // small basis records packed into one page

constexpr int kOffWr = kSlots * kSlotBytes;                     // W_r, 4 swizzled boxes (32 KB)
constexpr int kOffScratch = kOffWr + kRouteDim * kHeadDim * 4;  // q (4 KB) + y (2 KB)
constexpr int kOffInfo = kOffScratch + 6144;                    // summary bias per span (float)
constexpr int kOffMisc = kOffInfo + kInfoCap * 4;
constexpr int kMiscBytes = 6144;
constexpr int kSmemBytes = kOffMisc + kMiscBytes;
constexpr int kCombineChunk = 32;                       // partials per bulk copy (133 KB)
constexpr int kCombineLOff = kOffWr - kMaxCgSmem * 8 * 4;  // [cg][8] floats below W_r
constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment

enum PageType : int {
  PG_ROUTE = 1, PG_INFO = 2, PG_FULL = 3, PG_SUM = 4, PG_EXP = 5, PG_END = 6, PG_EXPM = 7,
  PG_SYNC = 8  // no data: every routing page of the CTA comes before it
};

// One basis record inside a PG_EXPM page (several small records per page).
struct RecInfo {
  int off;  // byte offset in the page
  int b, rk, rv;
};

struct PageDesc {
  int type;
  int n;       // rows / spans / body tokens / records in this page
  int a;       // first row / first span ordinal / first body token
  int rk, rv;  // expanded span: ranks
  int flag;    // PG_ROUTE: routing page index within the CTA
  int off_a;   // PG_EXP: byte offset of the key part (header..Vt_K) or -1
  int off_uk;  // PG_EXP: byte offset of U_K rows [a, a+n)
  int off_uv;  // PG_EXP: byte offset of U_V rows [a, a+n)
  int off_b;   // PG_EXP: byte offset of the value part (sigma_V..Vt_V) or -1
  int part;    // PG_EXP: part index of the record
  int b;       // PG_EXP: body tokens of the record
  long long src;  // PG_EXP: the record's byte offset from the store base
};

struct DecodeParams {
  CUtensorMap tm_kfull, tm_vfull, tm_ksum, tm_vsum, tm_sroute, tm_wr;
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
  ExpEntry* entries;     // fused: by span ordinal; list mode: compact, in list order
  uint64_t* pmask;       // fused: [group][cta][routing page] expanded-span bit masks
  int64_t* pbytes;       // fused: [group][cta][routing page] record bytes of those spans
  const uint16_t* info;  // list mode: per-span info written by the prep kernel
  Partial* partials;
  int B, Hq, Hkv, G, n_sink, n_recent, max_spans, cap_full, cg;
  float scale_log2;
  int fused;
  int rank_lim;  // largest record rank the kernel instance handles (16 KS)
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

template <int KS>
__global__ void decode_kernel(const __grid_constant__ DecodeParams P);
__global__ void prep_list_kernel(const PrepParams P);

// Host-side handles of the decode kernel instances (ranks up to 16 KS).
const void* decode_kernel_fn_ks1();
const void* decode_kernel_fn_ks2();
const void* decode_kernel_fn_ks3();
const void* decode_kernel_fn_ks4();

// Fixed-part split: CTA j of cg takes an equal share of the full-resolution
// rows and an equal share of the spans (routing summaries and summary rows),
// so routing is spread over all CTAs of a KV head.  Span boundaries are
// rounded up to multiples of 8 so that every per-span array slice starts
// 16-byte aligned.  32-bit arithmetic: the host rejects shapes with
// (2 (n_sink + n_recent) + 5 max_spans) * 256 >= 2^31.  (fused: unused, the
// split is the same in both modes.)
__host__ __device__ inline void fixed_range(int j, int cg, int n_full, int n_sp, int fused,
                                            int& f0, int& f1, int& k0, int& k1) {
  (void)fused;
  f0 = n_full * j / cg;
  f1 = n_full * (j + 1) / cg;
  auto kpos = [&](int jj) -> int {
    const int v = ((n_sp * jj / cg) + 7) & ~7;
    return v < n_sp ? v : n_sp;
  };
  k0 = kpos(j);
  k1 = kpos(j + 1);
}

// Boundary j of cg equal shares of T bytes (monotone in j, 0 at j = 0, T at
// j = cg); every CTA evaluates the same expression, so the shares tile [0, T).
__host__ __device__ inline long long byte_split(long long T, int j, int cg) {
  if (j >= cg) return T;
  return (long long)((double)T * j / cg);
}

struct SmemMisc {
  PageDesc desc[kSlots];
  RecInfo rec[kSlots][kMaxRecPerPage];
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  uint64_t wr_bar;   // W_r boxes landed (fused mode)
  uint64_t cmb_bar;  // last CTA of a KV head: a chunk of partials landed
  unsigned long long rmask[kMaxRoutePages];  // expanded spans per routing page (bit i: span a+i)
  long long rbytes[kMaxRoutePages];          // their record bytes
  int is_last;
  uint32_t warm[kConsumerWarps];  // sink of the instruction-cache warm-up pass
  float theta[8];
  int pre_n[kMaxCgSmem + 1];                 // expanded spans before CTA jj (exclusive prefix)
  long long pre_b[kMaxCgSmem + 1];           // their record bytes
  // warp w is loading and consuming a record larger than a page: set by the
  // producer when it hands the record over, cleared by warp w after its last part
  alignas(16) int sp_busy[kConsumerWarps];
};
static_assert(sizeof(SmemMisc) <= kMiscBytes, "misc smem");

constexpr uint32_t kWaitLimit = 1u << 24;  // bounded mbarrier polls (~1-2 s at most)
constexpr uint32_t kSpinLimit = 1u << 22;  // bounded polls of global counters (~2-3 s)

__device__ __forceinline__ uint8_t* slot_ptr(uint8_t* smem, int slot) {
  return smem + slot * kSlotBytes;
}

// Per-warp ring position (slot index within the warp's two, phase bit).
struct Ring {
  int s = 0;
  uint32_t phase = 0;
};

__device__ __forceinline__ void ring_advance(Ring& r) {
  if (++r.s == kSlotsPerWarp) {
    r.s = 0;
    r.phase ^= 1u;
  }
}

__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// U rows per middle part of a record larger than a page (multiple of 16).
__device__ __forceinline__ int split_rows(int rK, int rV) {
  const int row_bytes = 2 * (r8(rK) + r8(rV));
  int rows = row_bytes > 0 ? (kPageData / row_bytes) & ~15 : 512;
  return rows > 512 ? 512 : rows;
}

// Parts of such a record: the key part, ceil(b / rows) U tiles, the value part.
__device__ __forceinline__ int split_nparts(int b, int rK, int rV) {
  const int rows = split_rows(rK, rV);
  return 2 + (b + rows - 1) / rows;
}

// Part `part` of the record at store offset src (b body tokens, ranks rK,
// rV) into `slot`, whose previous page has been consumed: its descriptor, the
// full barrier armed with its bytes, then its one or two copies.  Issued by
// one thread (the producer for part 0, the consuming warp for the others).
__device__ __forceinline__ void issue_split_part(uint8_t* smem, SmemMisc* ms,
                                                 const DecodeParams& P, int slot, int part, int b,
                                                 int rK, int rV, long long src) {
  const RecordLayout L = record_layout(b, rK, rV);
  const int np = split_nparts(b, rK, rV);
  PageDesc d{};
  d.type = PG_EXP;
  d.rk = rK;
  d.rv = rV;
  d.off_a = -1;
  d.off_b = -1;
  d.part = part;
  d.b = b;
  d.src = src;
  int64_t s0 = 0, s1 = 0;
  uint32_t n0 = 0, n1 = 0;
  if (part == 0) {  // header, sigma_K, g_K, Vt_K
    d.off_a = 0;
    n0 = uint32_t(L.uk);
  } else if (part < np - 1) {  // U_K and U_V rows of one tile
    const int rows = split_rows(rK, rV);
    const int i0 = (part - 1) * rows;
    d.n = (b - i0) < rows ? (b - i0) : rows;
    d.a = i0;
    d.off_uv = 2 * d.n * r8(rK);
    s0 = L.uk + 2 * int64_t(i0) * r8(rK);
    n0 = uint32_t(d.off_uv);
    s1 = L.uv + 2 * int64_t(i0) * r8(rV);
    n1 = uint32_t(2 * d.n * r8(rV));
  } else {  // sigma_V, g_V, Vt_V
    d.off_b = 0;
    s0 = L.vpart;
    n0 = uint32_t(L.total - L.vpart);
  }
  ms->desc[slot] = d;
  mbar_arrive_expect_tx(&ms->full[slot], n0 + n1);
  uint8_t* pg = slot_ptr(smem, slot);
  const uint8_t* rec = P.store + src;
  const uint64_t pol = policy_evict_first();
  if (n0) bulk_g2s_hint(pg, rec + s0, n0, &ms->full[slot], pol);
  if (n1) bulk_g2s_hint(pg + n0, rec + s1, n1, &ms->full[slot], pol);
}

}  // namespace sekv
