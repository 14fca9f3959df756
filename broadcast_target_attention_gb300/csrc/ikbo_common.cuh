// Shared definitions of the IKBO target-attention kernels (sm_103a).
#pragma once

#include <cstdint>

namespace ikbo {

// Rows of one query tile: the M extent of the tcgen05 MMA.  A tile holds the
// query tokens of up to floor(128 / Lq) candidates of ONE user, so that all
// of them share every K/V tile the CTA streams ("In-Kernel Broadcast
// Optimization", §3.2: one CTA issues several candidates of the same user
// to fill the MMA M extent).
constexpr int kTileM = 128;

// Bits of the per-device error word.
constexpr int kErrIndex = 1;    // cand_to_user value outside [0, n_user)
constexpr int kErrOffsets = 2;  // user_offsets[0] != 0, or decreasing
constexpr int kErrTimeout = 4;  // a bounded wait ran out
constexpr int kErrLayout = 8;   // the kernel found its launch unusable (shared-memory alignment)

// One unit of work of the attention kernel: a query tile of one user and one
// head, against one contiguous range of that user's keys.  The tile holds
// either candidates' queries (q_row = -1) or, in a fused self + target call,
// up to 128 rows of the user's own sequence (q_user rows q_row ..
// q_row + n_cand - 1).
struct WorkItem {
  int32_t user;        // user index
  int32_t head;        // head index
  int32_t cand_begin;  // first position in the grouped candidate order
  int32_t n_cand;      // candidates in this tile (<= cands per tile); sequence rows of a self tile
  int32_t kv_begin;    // first key row in k/v (absolute, = user_offsets[u] + split start)
  int32_t kv_len;      // keys in this item (> 0)
  int32_t unit;        // split-combine unit, or -1 when the item covers all keys
  int32_t unit_first;  // first item index of the unit (its n_split items are consecutive)
  int32_t q_row;       // self-attention tile: its first row of q_user / out_user; else -1
  int32_t n_split;     // parts the unit's keys are cut into: key-interleaved kernel, chunks on as many
                       // CTAs (1 = the item covers all keys); two-tile kernel, 2 = a user's only query
                       // tile, its keys interleaved over the two warpgroups
};
static_assert(sizeof(WorkItem) == 40, "WorkItem layout");

struct PlanHeader {
  int32_t n_items;       // work items written
  int32_t sorted;        // 1: cand_to_user non-decreasing, grouped order == candidate order
  int32_t total_keys;    // T = user_offsets[n_user]
  int32_t split_tiles;   // key tiles per split item (0 = no splitting)
  int32_t work_counter;  // dynamic scheduler: next item to take
  int32_t n_units;       // split-combine units
  int32_t error;         // error bits found by the planner (0 = ok)
  int32_t pad;
};

// Per-unit record of a split (user, head, query tile): how many items, and
// the arrival counter the last-arriving CTA detects itself with.
struct UnitInfo {
  int32_t n_split;
  int32_t arrived;
};

// Planner parameters (host -> planning kernel).
struct PlanParams {
  const int32_t* cand_to_user;
  const int32_t* user_offsets;
  int64_t n_cand;
  int64_t n_user;
  int32_t H;
  int32_t cands_per_tile;   // floor(128 / Lq)
  int32_t block_n;          // keys per K/V tile
  int32_t num_sms;          // SMs of the device
  int32_t max_items;        // capacity of the work list
  int32_t max_split_items;  // capacity of the split partial buffers
  int32_t max_units;        // capacity of UnitInfo
  int32_t allow_split;      // 1: split key ranges when units are few (SIMT kernel); 0: never
  // outputs (workspace)
  PlanHeader* header;
  WorkItem* items;
  UnitInfo* units;
  int32_t* perm;            // [n_cand] grouped order -> candidate (only when unsorted)
  int32_t* cand_start;      // [n_user + 1] first grouped position of each user
  int32_t* scratch;         // [3 * n_user + 2] per-user counters, order and prefixes
  int* err_word;            // per-device error word
  // multi-level call: cand_to_user holds item_to_vendor; the planner first writes every
  // item's user, vendor_to_user[item_to_vendor[i]] (or -1 when a value is out of range),
  // to item_user [n_cand] and plans from that
  const int32_t* vendor_to_user;
  int64_t n_vendor;
  int32_t* item_user;
};

// Parameters shared by the attention kernels (host -> device).
struct AttnParams {
  const uint16_t* q;        // bf16 [n_cand, H, Lq, D]
  const uint16_t* k;        // bf16 [T, H, D]
  const uint16_t* v;        // bf16 [T, H, D]
  uint16_t* out;            // bf16 [n_cand, H, Lq, D]
  int64_t n_cand;
  int32_t H;
  int32_t Lq;
  float scale_log2;         // scale * log2(e): scores are kept in base 2
  int32_t max_items;        // grid-stride bound (items beyond header->n_items are skipped)
  const PlanHeader* header;
  const WorkItem* items;
  UnitInfo* units;
  const int32_t* perm;      // grouped position -> candidate, used when header->sorted == 0
  float* partial_o;         // [max_split_items, 128, D] unnormalised O of split items
  float2* partial_ml;       // [max_split_items, 128] (running max m in base 2, row sum l)
  int* err_word;
  const void* kmap;         // K/V tensor maps (device copies patched by the planner)
  const void* vmap;
  uint64_t timeout_ns;      // bound of every wait on another warp or the TMA/MMA units
  int32_t qbox;             // candidates per Q box of the sorted-order tensor map
  int32_t debug_flags;      // test hook: 1 = never arm the Q barrier (exercises the timeout path)
  uint64_t* trace;          // optional %globaltimer stamps [trace_ctas][kTraceItems][kTracePoints], or null
  int32_t trace_ctas;       // CTAs the trace buffer has room for (the SMs): CTAs past them are not traced
  // in-kernel planning (tcgen05 kernel, "fused" mode)
  int32_t fused;            // 1: every CTA plans from the index tensors itself; 0: read `items`
  int32_t cands_per_tile;
  const int32_t* user_offsets;
  const int32_t* cand_to_user;
  int64_t n_user;
  WorkItem* cta_items;      // fused: [grid][max_cta_items] this CTA's items
  int32_t max_cta_items;
  int32_t* perm_ws;         // fused, unsorted input: grouped position -> candidate
  CUtensorMap* map_slots;   // [grid][map_stride] tensor maps written on the device: K and V with the
                            // row count T (fused), then per work item a V copy bounded at its user's end
  int32_t map_stride;       // map slots per CTA: 2 + the most work items a CTA takes
  // fused self + target attention (one-tile tcgen05 kernel, in-kernel planning)
  const uint16_t* q_user;   // bf16 [T, H, D] queries of the user sequence, or null (target only)
  uint16_t* out_user;       // bf16 [T, H, D]
  int64_t total_rows;       // T as the caller gave it; user_offsets[n_user] must equal it
  int32_t exact_rows;       // 1: the K/V maps were encoded with the row count T (no tail copy)
  // multi-level call (user -> vendor -> item): cand_to_user holds item_to_vendor and an
  // item's user is vendor_to_user[item_to_vendor[i]], looked up while planning; null otherwise
  const int32_t* vendor_to_user;
  int64_t n_vendor;
  // key-interleaved kernel: a unit cut into key-range chunks on several CTAs
  // is merged by its first chunk from the others' partial results
  float4* ab_partial_o;     // [grid][D / 4][128] O / l of every chunk, 16-byte column groups row-minor
  float* ab_partial_lse;    // [grid][128] log-sum-exp (base 2) of every chunk's rows
  unsigned long long* ab_flags;   // [grid] a chunk's partial is complete: ab_marker
  unsigned long long ab_marker;   // non-zero, unique to the call
  // two-tile kernel with Cluster Launch Control (clc = 1): one CTA per unit of
  // work; a running CTA takes over CTAs that have not started.  Per SM a slot
  // of clc_slot_bytes: the plan's user tables (offsets, first candidates,
  // units before each rank, users by rank; n_user + 1 ints each), then from
  // clc_map_offset one bounded V map per user.
  int32_t clc;
  int32_t clc_slot_bytes;
  int32_t clc_map_offset;
  uint8_t* clc_slots;
};

// In-kernel timeline tracing (ikbo_set_trace): the first kTraceItems items of
// every CTA record %globaltimer (ns) at these points.
constexpr int kTraceItems = 4;
constexpr int kTracePoints = 16;
enum TracePoint {
  kTrCtaStart = 0,      // after the prologue (item slot 0 only)
  kTrProdItem = 1,      // producer starts the item
  kTrProdIssued = 2,    // producer issued every load of the item
  kTrMmaQ = 3,          // MMA warp saw the Q tile
  kTrMmaFirstS = 4,     // first S MMA issued
  kTrMmaLastPV = 5,     // last PV MMA issued
  kTrSmS0 = 6,          // softmax saw the first S
  kTrSmLastP = 7,       // softmax handed over the last P
  kTrEpiO = 8,          // epilogue: O complete in TMEM
  kTrEpiStored = 9,     // epilogue: output / partial stored
  kTrArrived = 10,      // split: arrival counted
  kTrMerged = 11,       // split: merge done (last arriver)
  kTrCtaEnd = 12,       // before teardown (item slot 0 only)
  kTrEpiSums = 13,      // epilogue, row 32: row sums of both halves combined
  kTrEpiSent = 14,      // epilogue, row 32: its warp's rows for the partner sent
  kTrEpiKept = 15       // epilogue, row 32: its warp's own rows stored
};

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  // round to nearest even; inputs here are finite
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pairs of fp32 (one instruction for two lanes of work, sm_100 and later).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

}  // namespace ikbo
