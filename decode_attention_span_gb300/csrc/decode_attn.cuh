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
// Structure.  Grid (cg, Hkv, B): CTA j of a (sequence, KV head) group owns
// an equal share of the group's spans.  It routes them, attends their
// summaries and rebuilds the expanded ones among them, so no CTA waits for
// another's routing.  Full-resolution rows (sinks, anchors, recent) need no
// routing: each CTA takes kStaticPages pages of them as its own, and the
// rest form a pool of the group from which CTAs take pages while they have
// nothing else to do, which evens out the CTAs' unequal record loads (the
// last CTA of a group to finish merges the group's partial softmax states).
//
// Eight warps per CTA, each its own producer and consumer: a warp owns a
// 24 KB arena of shared memory, claims work items (expanded records first,
// then the CTA's own pages: full-resolution rows, then summary rows, then
// pages from the group's pool), lands them in its arena with TMA (tensor
// copies with 128B swizzle for row and routing pages, 1-D bulk copies for
// basis records), and consumes them in issue order, keeping up to kMaxItems
// in flight.  Each
// warp keeps its own online-softmax state (query heads of the GQA group as
// the M rows of mma.sync; keys, tokens or ranks as N); the eight states and
// then the CTAs' states are merged at the end.
#pragma once

#include "sekv_common.cuh"

namespace sekv {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kGran = 1024;                   // arena granule (TMA swizzle alignment)
constexpr int kArenaGran = 25;                // arena of one warp, in granules
constexpr int kArenaBytes = kArenaGran * kGran;
constexpr int kMaxItems = 2;                  // items in flight per warp (main loop)
constexpr int kSlots = 4;                     // item slots (descriptor + mbarrier) per warp
constexpr int kRows = 16;                     // rows per summary page (one mma tile)
constexpr int kRowHalf = kRows * 128;         // one 128-byte half of a summary page's rows (2 KB)
constexpr int kRowPageBytes = 4 * kRowHalf;   // K and V, both halves (8 KB)
constexpr int kFullRows = 32;                 // rows per full-resolution page (two tiles)
constexpr int kFullHalf = kFullRows * 128;    // one 128-byte half of its rows (4 KB)
constexpr int kFullPageBytes = 4 * kFullHalf; // K and V, both halves (16 KB)
constexpr int kRouteSpans = 32;               // spans per routing page
constexpr int kRoutePageBytes = kRouteSpans * 256;  // 8 KB
constexpr int kSpanCap = 512;                 // spans of one CTA (bias cache, entries)
constexpr int kMaxRoutePages = kSpanCap / kRouteSpans;
constexpr int kWholeMax = 25600;              // records up to this size land whole (a whole arena)
constexpr int kTileMax = 24576;               // U-row tiles of larger records
constexpr int kMaxCg = 256;                   // CTAs per (sequence, KV head) group
constexpr int kStaticPages = 1;               // full-resolution pages each CTA owns
constexpr int kPoolClaim = 1;                 // pages per claim from the group's pool
constexpr int kMergeChunk = 32;               // partials per bulk copy in the merge
constexpr int kPrologueItems = 3;             // items per warp issued before the query

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffArena = 0;
constexpr int kOffQfrag = kWarps * kArenaBytes;          // query A fragments (2 KB)
constexpr int kOffQf = kOffQfrag + 2048;                 // query as f32 [8][128] (4 KB)
constexpr int kOffY = kOffQf + 4096;                     // y = W_r q, f32 [8][64] (2 KB)
constexpr int kOffBias = kOffY + 2048;                   // summary bias per span (2 KB)
constexpr int kOffEntries = kOffBias + kSpanCap * 4;     // expanded records (8 KB)
constexpr int kOffCmask = kOffEntries + kSpanCap * 16;   // multi-query: columns expanding each span
constexpr int kOffMisc = kOffCmask + kSpanCap;
constexpr int kMiscBytes = 4096;
constexpr int kSmemBytes = kOffMisc + kMiscBytes;
constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
// Routines that read a record read up to 16 KB past the end of its key part
// (padded rank rows, masked in registers): the smem after the arenas covers it.
static_assert(kSmemBytes - kOffQfrag >= 16 * 1024 + 1024, "over-read margin");
static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");

enum ItemType : int {
  IT_ROUTE = 1,  // routing summaries of kRouteSpans spans (consumed before the barrier)
  IT_FULL = 2,   // kFullRows full-resolution rows (K and V), the CTA's own or from the pool
  IT_SUM = 3,    // kRows summary rows (K and V) of unexpanded spans
  IT_REC = 4,    // one whole basis record
  IT_KEY = 5,    // key part of a split record (header, sigma_K, g_K, Vt_K)
  IT_UT = 6,     // U_K and U_V rows of one tile of a split record
  IT_VAL = 7,    // value part of a split record (sigma_V, g_V, Vt_V)
};

struct Item {      // one landed (or landing) work item of a warp, 32 bytes
  int type;
  int n;           // rows / spans / tokens of a U tile / body of a record
  int a;           // first row / first span; records: the query columns that expand the span
  int rk, rv;      // record ranks
  int boff;        // byte offset of the item's data from the CTA's arena base
  int end;         // the warp's arena granule counter at the item's end
  int uv;          // IT_UT: byte offset of the U_V rows from the item's data
};

// One expanded span of the CTA, 16 bytes, with what the issue logic needs
// worked out when the entry is made (by the routing lanes, in parallel).
struct RecEntry {
  int off_lo, off_hi;  // byte offset of its record from `store`
  int body;            // |S| | columns expanding the span << 16 | parts << 24 (0: skipped)
  int rank;            // rK | (U rows per tile / 16) << 8 | rV << 16
};

struct DecodeParams {
  CUtensorMap tm_kfull, tm_vfull, tm_ksum, tm_vsum, tm_sroute;
  const int32_t* n_spans;
  const int32_t* n_tail;   // [B] full-resolution rows after the anchors, or null: n_recent
  const int32_t* body_len;
  const int64_t* rec_off;
  const int32_t* rec_rank;
  const uint8_t* store;          // base that record offsets refer to (store or staging)
  const __nv_bfloat16* q;
  const float* W_r;              // fused mode
  const float* theta;            // fused mode
  const int32_t* list;           // list mode: ascending expansion lists [g][max_spans]
  const int32_t* list_n;         // list mode: their lengths [g]
  const int64_t* staged_off;     // list mode, optional: record offsets [g][max_spans]
  float* out;
  float* lse;
  int32_t* expanded_out;         // fused mode, optional
  int32_t* n_expanded_out;
  int32_t* status;
  GroupState* groups;
  int32_t* cta_n;                // [g][cg] expanded spans per CTA (fused, list output)
  int32_t* cta_list;             // [g][max_spans] them, ascending within each CTA's share
  float* partials;               // [g][cg] of 16 + G*128 floats (m[8], l[8], o[G][128])
  // G: query columns of a group, mma N -- the group's heads, or (multi-query
  // decode) nq query tokens x hpg heads; column h is token h / hpg, head h % hpg
  int B, Hq, Hkv, G, n_sink, n_recent, max_spans, cg;
  int nq, hpg;    // query tokens of this launch; heads per group (column h: token h / hpg)
  int nq_all;     // query tokens per sequence in q, out and lse (their sequence stride)
  float scale_log2;
  int fused;
  int rank_lim;                  // largest record rank the kernel instance handles (16 KS)
  unsigned long long wait_ns;    // limit of a parked wait for an item (SEKV_FLAG_SHORT_WAITS: 0)
};

// KS: rank k-steps of 16 (ranks up to 16 KS); MQ: multi-query decode (query
// columns of several tokens, per-token expansion masks), a separate instance
// so that the one-token step carries none of its masking
template <int KS, bool MQ>
__global__ void decode_kernel(const __grid_constant__ DecodeParams P);

// Host-side handles of the decode kernel instances (ranks up to 16 KS).
const void* decode_kernel_fn_ks1(bool mq);
const void* decode_kernel_fn_ks2(bool mq);
const void* decode_kernel_fn_ks3(bool mq);
const void* decode_kernel_fn_ks4(bool mq);

// Span share [k0, k1) of CTA j of cg.  Boundaries are rounded up to
// multiples of 8 so that every per-span array slice starts 16-byte aligned.
// 32-bit arithmetic: the host rejects shapes with
// (2 (n_sink + n_recent) + 5 max_spans) * 256 >= 2^31.
__host__ __device__ inline void span_range(int j, int cg, int n_sp, int& k0, int& k1) {
  auto kpos = [&](int jj) -> int {
    const int v = ((n_sp * jj / cg) + 7) & ~7;
    return v < n_sp ? v : n_sp;
  };
  k0 = kpos(j);
  k1 = kpos(j + 1);
}

// Everything a CTA derives from its block index (computed once, kept in
// shared memory).
struct Ctx {
  int g, j, b, c;
  int n_sp;     // spans of the sequence
  int k0, k1;   // the CTA's spans
  int n_full;   // full-resolution rows of the group
  int n_fp;     // their pages
  int own0;     // first of the CTA's own full-resolution pages
  int n_own;    // how many it owns (kStaticPages, fewer at the end)
  int pool0;    // first page of the group's pool (the pages no CTA owns)
  int n_fixed;  // the CTA's own full-resolution pages + its summary pages
  int n_rp;     // routing pages (fused mode)
  long long gs; // g * max_spans
  long long bs; // b * max_spans
};

// Issue state of one warp, in shared memory (lane 0 issues; every lane reads
// ni / nd / ok after a __syncwarp).
struct WarpQ {
  int head, tail;   // arena granule counters (monotone)
  int ni, nd;       // items issued / consumed
  int pk;           // pending claim: 0 none, 1 own page, 2 record, 3 pool pages
  int pidx;         // its index (own page, record entry, first pool page)
  int ppart, pnp;   // record: next part, parts; pool: next page, pages
  int fixed_out;    // own pages exhausted
  int rec_out;      // record queue exhausted
  int pool_out;     // the group's pool exhausted
  int ok;           // no wait has run out
};

struct SmemMisc {
  Ctx ctx;
  WarpQ wq[kWarps];
  Item desc[kWarps][kSlots];
  uint64_t bar[kWarps][kSlots];
  uint64_t cmb_bar;        // last CTA of a group: a chunk of partials landed
  unsigned int pmask[kMaxRoutePages];  // fused: expanded spans per routing page
  float theta[8];
  int n_front;             // expanded records in parts, from the front of the entries
  int n_back;              // the other expanded records, from the back of the entries
  int rec_next;            // record queue head
  int fixed_next;          // fixed-page queue head
  int is_last;
  int list_base;           // list mode: first list entry of this CTA's share
};
static_assert(sizeof(SmemMisc) <= kMiscBytes, "misc smem");

constexpr uint32_t kWaitLimit = 1u << 24;  // bounded mbarrier polls (~1-2 s at most)
constexpr unsigned long long kMergeWaitNs = 2000000000ull;  // bounded wait for the partials

// U rows per tile of a split record (a multiple of 16, at most 512).
__host__ __device__ inline int split_rows(int rK, int rV) {
  const int row_bytes = 2 * (r8(rK) + r8(rV));
  int rows = row_bytes > 0 ? (kTileMax / row_bytes) & ~15 : 512;
  return rows > 512 ? 512 : (rows < 16 ? 16 : rows);
}

// Parts of a record: 1 if it lands whole, else the key part, ceil(b / rows)
// U tiles and the value part.
__host__ __device__ inline int record_parts(int b, int rK, int rV) {
  if (record_bytes(b, rK, rV) <= kWholeMax) return 1;
  const int rows = split_rows(rK, rV);
  return 2 + (b + rows - 1) / rows;
}

// Entry slot of the e-th record of a CTA's queue: the n_front records in
// parts first (from the front of the entries), then the others (from the back).
__host__ __device__ inline int rec_slot(int e, int n_front) {
  return e < n_front ? e : kSpanCap - 1 - (e - n_front);
}

}  // namespace sekv
