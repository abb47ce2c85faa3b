// Internal declarations shared by the translation units of libthdattn.so:
// workspace layout, the per-work-item geometry of the emulated ring, and the
// host-side launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/thd_attn.h"

namespace thd {

constexpr int kTile = 128;          // rows of a query tile and of a key/value tile
constexpr int kPlanThreads = 1024;  // threads of the single-CTA planner
constexpr int kCostBins = 4096;     // counting-sort bins for the longest-first order

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }

// ---------------------------------------------------------------- workspace
// Effective metadata written by the planner (after the pad decision):
//   eff[0][*] = cu_q, eff[1][*] = pad_q, eff[2][*] = cu_kv, eff[3][*] = pad_kv
struct WsLayout {
  size_t eff = 0;       // int32 [4][B+1]
  size_t tile_off = 0;  // int32 [B+1]
  size_t counters = 0;  // int32 [64]: [0] number of schedule entries
  size_t items = 0;     // int4 [item_cap]
  // backward only: the query-tile schedule of the dQ pass (its own planner
  // outputs), Delta = rowsum(dO * O) and lse in log2 units
  size_t tile_off_q = 0;  // int32 [B+1]
  size_t counters_q = 0;  // int32 [64]
  size_t items_q = 0;     // int4 [item_cap_q]
  size_t delta = 0;       // fp32 [Hq][T_q]
  size_t lse2 = 0;        // fp32 [Hq][T_q], lse * log2(e)
  size_t total = 0;
  int item_cap = 0;
  int item_cap_q = 0;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int B, int64_t T_q, int64_t T_kv, int Hq, int D, int cp, bool bwd) {
  WsLayout w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.eff = take(sizeof(int32_t) * 4 * (size_t)(B + 1));
  w.tile_off = take(sizeof(int32_t) * (size_t)(B + 1));
  w.counters = take(sizeof(int32_t) * 64);
  // query schedule: rank-local query tiles; key schedule: chunk-aligned key
  // tiles.  Both are bounded by rows/128 + (one partial tile per chunk).
  const int64_t cap_q = T_q / kTile + (int64_t)cp * B + 1;
  const int64_t cap_kv = T_kv / kTile + (int64_t)2 * cp * B + 1;
  w.item_cap = (int)(bwd ? cap_kv : cap_q);
  w.items = take(sizeof(int32_t) * 4 * (size_t)w.item_cap);
  if (bwd) {
    w.item_cap_q = (int)cap_q;
    w.tile_off_q = take(sizeof(int32_t) * (size_t)(B + 1));
    w.counters_q = take(sizeof(int32_t) * 64);
    w.items_q = take(sizeof(int32_t) * 4 * (size_t)cap_q);
    w.delta = take(sizeof(float) * (size_t)Hq * (size_t)T_q);
    w.lse2 = take(sizeof(float) * (size_t)Hq * (size_t)T_q);
  }
  (void)D;
  w.total = off;
  return w;
}

// ---------------------------------------------------------------- geometry
// One sequence's view after the pad decision.
struct SeqGeom {
  int q_off, kv_off;  // buffer row of position 0
  int Lq, Lkv;        // valid lengths
  int cbq, cbkv;      // chunk lengths (padded / (2 cp))
  int koff;           // causal masks: query i sees key j iff j <= i + koff
};

// Causal modes (the `causal` argument of the entry points).
constexpr int kCausalNone = THD_CAUSAL_NONE;
constexpr int kCausalTopLeft = THD_CAUSAL_TOP_LEFT;          // j <= i; equal query and key lengths
constexpr int kCausalBottomRight = THD_CAUSAL_BOTTOM_RIGHT;  // j <= i + Lkv - Lq: last query sees last key

__device__ inline SeqGeom seq_geom(const int32_t* eff, int B, int b, int cp, int causal) {
  const int32_t* cu_q = eff;
  const int32_t* pad_q = eff + (B + 1);
  const int32_t* cu_kv = eff + 2 * (B + 1);
  const int32_t* pad_kv = eff + 3 * (B + 1);
  SeqGeom g;
  g.q_off = pad_q[b];
  g.kv_off = pad_kv[b];
  g.Lq = cu_q[b + 1] - cu_q[b];
  g.Lkv = cu_kv[b + 1] - cu_kv[b];
  g.cbq = (pad_q[b + 1] - pad_q[b]) / (2 * cp);
  g.cbkv = (pad_kv[b + 1] - pad_kv[b]) / (2 * cp);
  g.koff = causal == kCausalBottomRight ? g.Lkv - g.Lq : 0;
  return g;
}

// Position (within the sequence) of rank r's rank-local query row p:
// rows [0, cb) are chunk r, rows [cb, 2cb) chunk 2cp-1-r.
__host__ __device__ inline int local_to_pos(int p, int r, int cb, int cp) {
  return p < cb ? r * cb + p : (2 * cp - 1 - r) * cb + (p - cb);
}

// Largest valid query position among rank-local rows [128 t, 128 t + 128)
// of rank r, or -1 when the tile holds no valid query.
__host__ __device__ inline int fwd_tile_qmax(const SeqGeom& g, int r, int t, int cp) {
  const int p0 = t * kTile, p1 = imin(p0 + kTile, 2 * g.cbq);
  int qmax = -1;
  // first half (chunk r)
  int a0 = p0, a1 = imin(p1, g.cbq);
  if (a0 < a1) {
    int last = imin(local_to_pos(a1 - 1, r, g.cbq, cp), g.Lq - 1);
    if (local_to_pos(a0, r, g.cbq, cp) <= last) qmax = imax(qmax, last);
  }
  // second half (chunk 2cp-1-r)
  a0 = imax(p0, g.cbq);
  a1 = p1;
  if (a0 < a1) {
    int last = imin(local_to_pos(a1 - 1, r, g.cbq, cp), g.Lq - 1);
    if (local_to_pos(a0, r, g.cbq, cp) <= last) qmax = imax(qmax, last);
  }
  return qmax;
}

// Number of 128-row key tiles of chunk c that a query tile with largest
// valid position qmax visits (tiles whose first key is past every query, or
// past the valid length, are skipped).
__host__ __device__ inline int fwd_chunk_tiles(const SeqGeom& g, int c, int qmax, bool causal) {
  if (qmax < 0) return 0;
  const int limit = causal ? imin(g.Lkv, qmax + g.koff + 1) : g.Lkv;
  const int start = c * g.cbkv;
  if (start >= limit) return 0;
  return imin(ceil_div(g.cbkv, kTile), ceil_div(limit - start, kTile));
}

// Ring step i of rank r holds the KV of rank s = (r - i) mod cp; its chunks
// are s and 2cp-1-s (in that order).
__host__ __device__ inline int ring_src(int r, int i, int cp) { return ((r - i) % cp + cp) % cp; }
__host__ __device__ inline int ring_chunk(int s, int e, int cp) { return e == 0 ? s : 2 * cp - 1 - s; }

// Key tiles one forward work item visits over ring steps [step_lo, step_hi).
__host__ __device__ inline int fwd_item_tiles(const SeqGeom& g, int r, int t, int cp, bool causal, int step_lo,
                                              int step_hi) {
  const int qmax = fwd_tile_qmax(g, r, t, cp);
  int n = 0;
  for (int i = step_lo; i < step_hi; ++i) {
    const int s = ring_src(r, i, cp);
    for (int e = 0; e < 2; ++e) n += fwd_chunk_tiles(g, ring_chunk(s, e, cp), qmax, causal);
  }
  return n;
}

// ---- one query tile's walk (forward and the dQ pass).  P is any params
// struct with items, eff, B, Hq, Hkv, cp, causal, step_lo, step_hi.
struct QItem {
  SeqGeom g;
  int b, r, t, h, kvh, qmax;
};

// Work item w -> (schedule entry, query head).  Items are ordered by groups
// of p.group_kv kv heads (outermost: while a group runs, its keys and values
// are what the CTAs read, so they stay in L2), then by schedule entry
// (longest first), then by the group's query heads (innermost: query heads
// that share a kv head run side by side).  Ungrouped (one group, group_kv ==
// Hkv) it is entry-major with every head innermost.  n_entries = schedule
// length.
// kGrouped is a compile-time choice: a runtime branch between the two maps
// here measured 8% slower in the forward kernel.
template <bool kGrouped, class P>
__device__ inline QItem q_item(const P& p, int n_entries, int w) {
  QItem it;
  int4 e;
  if constexpr (kGrouped) {
    const int hg = p.group_kv * (p.Hq / p.Hkv);  // query heads per group
    const int per = n_entries * hg;               // items per group
    const int grp = w / per, rem = w - grp * per;
    e = p.items[rem / hg];
    it.h = grp * hg + rem % hg;
  } else {  // one group: entry-major, heads innermost
    (void)n_entries;
    e = p.items[w / p.Hq];
    it.h = w % p.Hq;
  }
  it.b = e.x;
  it.r = e.y;
  it.t = e.z;
  it.kvh = it.h / (p.Hq / p.Hkv);
  it.g = seq_geom(p.eff, p.B, it.b, p.cp, p.causal);
  it.qmax = fwd_tile_qmax(it.g, it.r, it.t, p.cp);
  return it;
}

// Calls f(c, j) for every key tile the item visits, in ring order: step i
// holds the KV of rank s = (r - i) mod cp, chunks s then 2cp-1-s.
template <class P, typename F>
__device__ inline void for_each_kv_tile(const QItem& it, const P& p, F&& f) {
  for (int i = p.step_lo; i < p.step_hi; ++i) {
    const int s = ring_src(it.r, i, p.cp);
    for (int e = 0; e < 2; ++e) {
      const int c = ring_chunk(s, e, p.cp);
      const int n = fwd_chunk_tiles(it.g, c, it.qmax, p.causal != 0);
      for (int j = 0; j < n; ++j) f(c, j);
    }
  }
}

// Columns (keys) of tile (c, j) any query of the item may see, rounded up to
// the MMA granularity of 16: the N of the item's S product and the K of the
// product that contracts over keys.
template <class P>
__device__ inline int q_tile_ncols(const QItem& it, const P& p, int c, int j) {
  const int j0 = c * it.g.cbkv + j * kTile;
  int n = imin(kTile, imin((c + 1) * it.g.cbkv - j0, it.g.Lkv - j0));
  if (p.causal) n = imin(n, it.qmax + it.g.koff - j0 + 1);
  return 16 * ceil_div(imax(n, 1), 16);
}

// ---- backward: key tile (chunk c, tile jk) of sequence b, and the query
// tiles (chunk qc, tile jq) that attend to it, walked in ring order: the KV of
// owner s is held by rank r = (s + i) mod cp at step i; rank r's query chunks
// are r and 2cp-1-r.
__host__ __device__ inline int chunk_owner(int c, int cp) { return c < cp ? c : 2 * cp - 1 - c; }

// [first, last] valid key positions of key tile (c, jk), or first > last.
__host__ __device__ inline void bwd_kv_range(const SeqGeom& g, int c, int jk, int& first, int& last) {
  first = c * g.cbkv + jk * kTile;
  last = imin(c * g.cbkv + imin((jk + 1) * kTile, g.cbkv), g.Lkv) - 1;
}
// Does query tile (qc, jq) hold a query that sees key position kv_first?
__host__ __device__ inline bool bwd_q_tile_visits(const SeqGeom& g, int qc, int jq, int kv_first, int kv_last,
                                                  bool causal) {
  if (kv_first > kv_last) return false;
  const int q0 = qc * g.cbq + jq * kTile;
  const int qlast = imin(qc * g.cbq + imin((jq + 1) * kTile, g.cbq), g.Lq) - 1;
  if (q0 > qlast) return false;
  return causal ? (qlast + g.koff >= kv_first) : true;
}
__host__ __device__ inline int bwd_item_qtiles(const SeqGeom& g, int c, int jk, int cp, bool causal) {
  int kf, kl;
  bwd_kv_range(g, c, jk, kf, kl);
  if (kf > kl) return 0;
  const int s = chunk_owner(c, cp);
  const int nq = ceil_div(g.cbq, kTile);
  int n = 0;
  for (int i = 0; i < cp; ++i) {
    const int r = (s + i) % cp;
    for (int e = 0; e < 2; ++e) {
      const int qc = e == 0 ? r : 2 * cp - 1 - r;
      for (int jq = 0; jq < nq; ++jq) n += bwd_q_tile_visits(g, qc, jq, kf, kl, causal) ? 1 : 0;
    }
  }
  return n;
}

// ---------------------------------------------------------------- planner
struct PlanParams {
  const int32_t* cu_q;
  const int32_t* cu_kv;
  const int32_t* pad_q;   // may be null
  const int32_t* pad_kv;  // may be null
  int B, cp, causal, pad_mode;
  int64_t rows_q, rows_kv;  // buffer rows
  int mode;                 // 0: partition only, 1: query-tile schedule, 2: key-tile schedule,
                            // 3: both (key tiles into items, query tiles into items_q)
  int step_lo, step_hi;     // ring steps the forward items cover (for the cost)
  int32_t* eff;             // [4][B+1]
  int32_t* cu_rank;         // optional partition outputs (q side)
  int32_t* cu_rank_padded;
  int32_t* cu_rank_half;
  int32_t* token_map;
  int64_t token_map_cap;
  int32_t* tile_off;  // [B+1]
  int32_t* counters;  // [64]
  int4* items;
  int item_cap;
  int32_t* tile_off_q;  // mode 3: the query-tile schedule's outputs
  int32_t* counters_q;
  int4* items_q;
  int item_cap_q;
  int32_t* dev_status;
};

// ---------------------------------------------------------------- kernels
struct FwdParams {
  const uint16_t* q;
  void* o;        // bf16 [T_q][Hq][D] (fused) or fp32 (one ring step)
  float* lse;     // [Hq][T_q]
  const int32_t* eff;
  const int4* items;
  const int32_t* counters;
  int32_t* claim;  // dynamic hand-out counter (zeroed by the planner)
  int32_t* dev_status;
  int B, Hq, Hkv, cp, causal;
  int group_kv;  // kv heads per locality group (divides Hkv)
  int64_t T_q;
  float scale_log2;  // softmax_scale * log2(e)
  int step_lo, step_hi;
  int test_stall;  // test hook: every thread waits for a barrier nothing completes
};

struct BwdParams {
  const uint16_t* q;
  const uint16_t* dout;
  const float* lse2;   // [Hq][T_q], lse * log2(e)
  const float* delta;  // [Hq][T_q]: Delta = rowsum(dO * O)
  uint16_t* dk;
  uint16_t* dv;
  const int32_t* eff;
  const int4* items;
  const int32_t* counters;
  int32_t* claim;  // dynamic hand-out counter (zeroed by the planner)
  int32_t* dev_status;
  int B, Hq, Hkv, cp, causal;
  int group_kv;  // kv heads per locality group (divides Hkv)
  int64_t T_q, dkv_rows;
  float scale, scale_log2;
  int test_stall;  // test hook: every thread waits for a barrier nothing completes
};

struct DqParams {
  const uint16_t* q;
  const uint16_t* dout;
  const float* lse2;   // [Hq][T_q], lse * log2(e)
  const float* delta;  // [Hq][T_q]: Delta = rowsum(dO * O)
  uint16_t* dq;       // bf16 [dq_rows][Hq][D]
  const int32_t* eff;
  const int4* items;  // the query-tile schedule
  const int32_t* counters;
  int32_t* claim;  // dynamic hand-out counter (zeroed by the planner)
  int32_t* dev_status;
  int B, Hq, Hkv, cp, causal;
  int group_kv;  // kv heads per locality group (divides Hkv)
  int64_t T_q, dq_rows;
  float scale, scale_log2;
  int step_lo, step_hi;  // always the whole ring
  int test_stall;  // test hook: every thread waits for a barrier nothing completes
};

// host launchers (each returns a cudaError_t)
cudaError_t launch_plan(const PlanParams& p, cudaStream_t st);
cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int D, bool step_mode,
                       bool dyn, int grid, cudaStream_t st);
cudaError_t launch_fwd_dual(const FwdParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int D, bool step_mode,
                            int grid, cudaStream_t st);
cudaError_t launch_bwd(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                       const CUtensorMap& tv, int D, bool grouped, int grid, cudaStream_t st);
cudaError_t launch_dq(const DqParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int D, bool grouped,
                      int grid, cudaStream_t st);
cudaError_t launch_lse_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part, int64_t T,
                             int H, int D, cudaStream_t st);
cudaError_t launch_lse_merge_bf16(float* o_acc, float* lse_acc, const uint16_t* o_part, const float* lse_part,
                                  int64_t T, int H, int D, cudaStream_t st);
cudaError_t launch_tail_zero(uint16_t* dq, uint16_t* dk, uint16_t* dv, int64_t dq_rows, int64_t dkv_rows, int Hq,
                             int Hkv, int D, const int32_t* pad_q_end, const int32_t* pad_kv_end,
                             const int32_t* dev_status, cudaStream_t st);
cudaError_t launch_bwd_prep(const uint16_t* o, const uint16_t* dout, const float* lse, float* delta, float* lse2,
                            const int32_t* eff, int B, int64_t T_q, int Hq, int D, const int32_t* dev_status,
                            cudaStream_t st);

int num_sms();
bool take_test_stall(int kernel_id);
int test_fwd_kernel();
void prof_before(int kernel_id, cudaStream_t st);
void prof_after(int kernel_id, cudaStream_t st);
void count_launch();

}  // namespace thd
