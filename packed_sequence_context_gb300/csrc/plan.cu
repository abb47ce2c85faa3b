// Metadata validation + pad detection (from values), the per-rank partition,
// the longest-first tile schedule, and the small HBM-bound kernels: LSE
// merge, gradient tail-zero and the backward preprocess (Delta, lse in log2
// units).
//
// Pages: [P2] TransformerEngine issue #3487 ("Describe the bug": the
// padding detector decides by object identity and get_cu_seqlens_on_cp_rank
// is called per ring step; THD dQ/dK/dV tail-zeroing launches work even with
// no tail; "Expected behavior": decide from values, stay graph-safe),
// [P3] "Hybrid / Hierarchical Context Parallel Skill" ("Contraintes
// requises": padded length divisible by 2 * cp_size).
#include <climits>
#include <cuda_bf16.h>

#include "common.cuh"

namespace thd {

// ------------------------------------------------------------------ helpers
// Exclusive scan over the 1024 threads of the block; `total` receives the sum.
__device__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int prefix = warp ? s_warp[warp - 1] : 0;
  total = s_warp[nwarps - 1];
  __syncthreads();
  return prefix + x - v;
}

// Largest b in [0, n] with a[b] <= x (a non-decreasing, a[0] <= x).
__device__ inline int upper_index(const int32_t* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ inline void set_err(int* s_err, int code) { atomicMin(s_err, code); }

// ------------------------------------------------------------------ planner
// The planner stages the effective metadata and tile offsets in shared memory
// when B + 1 <= kPlanSmemSeqs.
constexpr int kPlanSmemSeqs = 1024;

// a3: one schedule.  Query-tile entries are rank-local query tiles (b, r, t);
// key-tile entries are chunk-aligned key tiles (b, c, jk).  Both are ordered
// longest-first (counting sort on the number of tiles visited).  `eff` and
// `toff` are where the planner reads the effective metadata and the tile
// offsets (shared memory when they fit); `tile_off` receives the offsets in
// the workspace.  Returns false when the schedule exceeds its capacity.
__device__ bool plan_schedule(const PlanParams& p, const int32_t* eff, int32_t* toff, int mode, int32_t* tile_off,
                              int32_t* counters, int4* items, int item_cap, int* s_warp, int* s_hist) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int B = p.B, cp = p.cp;

  int carry = 0;
  for (int base = 0; base < B; base += nt) {
    const int b = base + tid;
    int n = 0;
    if (b < B) {
      SeqGeom g = seq_geom(eff, B, b, cp, p.causal);
      n = mode == 1 ? cp * ceil_div(2 * g.cbq, kTile) : 2 * cp * ceil_div(g.cbkv, kTile);
    }
    int tot;
    const int ex = block_exclusive_scan(n, s_warp, tot);
    if (b < B) {
      tile_off[b] = carry + ex;
      toff[b] = carry + ex;
    }
    carry += tot;
  }
  if (tid == 0) {
    tile_off[B] = carry;
    toff[B] = carry;
  }
  const int total = carry;
  if (total > item_cap) {
    if (tid == 0) *p.dev_status = THD_DEV_ERR_CAPACITY;
    return false;
  }
  for (int i = tid; i < kCostBins; i += nt) s_hist[i] = 0;
  __syncthreads();
  auto entry = [&](int w, int& b, int& x, int& y, int& cost) {
    b = upper_index(toff, B, w);
    // skip empty sequences that share the same offset
    while (b < B && toff[b + 1] <= w) ++b;
    SeqGeom g = seq_geom(eff, B, b, cp, p.causal);
    const int rem = w - toff[b];
    if (mode == 1) {
      const int per_r = ceil_div(2 * g.cbq, kTile);
      x = rem / per_r;
      y = rem % per_r;
      cost = fwd_item_tiles(g, x, y, cp, p.causal != 0, p.step_lo, p.step_hi);
    } else {
      const int per_c = ceil_div(g.cbkv, kTile);
      x = rem / per_c;
      y = rem % per_c;
      cost = bwd_item_qtiles(g, x, y, cp, p.causal != 0);
    }
  };
  for (int w = tid; w < total; w += nt) {
    int b, x, y, cost;
    entry(w, b, x, y, cost);
    atomicAdd(&s_hist[kCostBins - 1 - imin(cost, kCostBins - 1)], 1);
  }
  __syncthreads();
  // exclusive scan of the histogram: 4 bins per thread
  {
    constexpr int per = kCostBins / kPlanThreads;
    int loc[per];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      loc[j] = s_hist[tid * per + j];
      sum += loc[j];
    }
    int tot;
    int ex = block_exclusive_scan(sum, s_warp, tot);
#pragma unroll
    for (int j = 0; j < per; ++j) {
      s_hist[tid * per + j] = ex;
      ex += loc[j];
    }
  }
  __syncthreads();
  for (int w = tid; w < total; w += nt) {
    int b, x, y, cost;
    entry(w, b, x, y, cost);
    const int pos = atomicAdd(&s_hist[kCostBins - 1 - imin(cost, kCostBins - 1)], 1);
    items[pos] = make_int4(b, x, y, cost);
  }
  if (tid == 0) {
    counters[0] = total;
    counters[1] = 0;  // the attention kernel's dynamic hand-out counter
  }
  return true;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
  __shared__ int s_err;
  __shared__ int s_pad[2];
  __shared__ int s_warp[32];
  __shared__ int s_hist[kCostBins];
  // effective metadata [4][B+1] and tile offsets [B+1], when B + 1 <= kPlanSmemSeqs
  __shared__ int32_t s_meta[5 * kPlanSmemSeqs];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int B = p.B, cp = p.cp;
  const bool meta_in_smem = B + 1 <= kPlanSmemSeqs;
  if (tid == 0) {
    s_err = INT_MAX;
    s_pad[0] = 0;
    s_pad[1] = 0;
  }
  __syncthreads();
  // a1: padding between sequences, decided from VALUES.
  if (p.pad_mode == -1) {
    for (int b = tid; b <= B; b += nt) {
      if (p.pad_q && p.pad_q[b] != p.cu_q[b]) s_pad[0] = 1;
      if (p.pad_kv && p.pad_kv[b] != p.cu_kv[b]) s_pad[1] = 1;
    }
  }
  __syncthreads();
  const int padq = p.pad_q ? (p.pad_mode == -1 ? s_pad[0] : p.pad_mode) : 0;
  const int padkv = p.pad_kv ? (p.pad_mode == -1 ? s_pad[1] : p.pad_mode) : 0;
  const int32_t* PQ = padq ? p.pad_q : p.cu_q;
  const int32_t* PK = padkv ? p.pad_kv : p.cu_kv;
  int32_t* eff = p.eff;
  for (int b = tid; b <= B; b += nt) {
    const int cq = p.cu_q[b], pq = PQ[b], ck = p.cu_kv[b], pk = PK[b];
    if (eff) {
      eff[b] = cq;
      eff[(B + 1) + b] = pq;
      eff[2 * (B + 1) + b] = ck;
      eff[3 * (B + 1) + b] = pk;
    }
    if (meta_in_smem) {
      s_meta[b] = cq;
      s_meta[(B + 1) + b] = pq;
      s_meta[2 * (B + 1) + b] = ck;
      s_meta[3 * (B + 1) + b] = pk;
    }
    if (b == 0 && (cq != 0 || pq != 0 || ck != 0 || pk != 0)) set_err(&s_err, THD_DEV_ERR_NONZERO_START);
    if (b < B) {
      const int Lq = p.cu_q[b + 1] - cq, Pq = PQ[b + 1] - pq;
      const int Lk = p.cu_kv[b + 1] - ck, Pk = PK[b + 1] - pk;
      if (Lq < 0 || Pq < 0 || Lk < 0 || Pk < 0) set_err(&s_err, THD_DEV_ERR_NOT_MONOTONE);
      else if (Lq > Pq || Lk > Pk) set_err(&s_err, THD_DEV_ERR_VALID_GT_PAD);
      else if (Pq % (2 * cp) != 0 || Pk % (2 * cp) != 0) set_err(&s_err, THD_DEV_ERR_NOT_DIVISIBLE);
      else if (p.causal == kCausalTopLeft && (Lq != Lk || Pq != Pk)) set_err(&s_err, THD_DEV_ERR_CAUSAL_LENGTHS);
    } else {
      if ((int64_t)pq > p.rows_q || (int64_t)pk > p.rows_kv) set_err(&s_err, THD_DEV_ERR_EXCEEDS_BUF);
      if (p.token_map && (int64_t)pq > p.token_map_cap) set_err(&s_err, THD_DEV_ERR_EXCEEDS_BUF);
    }
  }
  __syncthreads();
  const int err = s_err == INT_MAX ? 0 : s_err;
  if (err) {
    if (tid == 0) *p.dev_status = err;
    return;
  }
  if (tid == 0) *p.dev_status = 0;

  // a2: per-rank partition (query side), every rank in this one launch.
  if (p.cu_rank || p.cu_rank_padded || p.cu_rank_half) {
    for (int r = tid; r < cp; r += nt) {
      int acc = 0, acc1 = 0, acc2 = 0;
      if (p.cu_rank) p.cu_rank[r * (B + 1)] = 0;
      if (p.cu_rank_half) {
        p.cu_rank_half[(r * 2 + 0) * (B + 1)] = 0;
        p.cu_rank_half[(r * 2 + 1) * (B + 1)] = 0;
      }
      for (int b = 0; b < B; ++b) {
        const int L = p.cu_q[b + 1] - p.cu_q[b];
        const int cb = (PQ[b + 1] - PQ[b]) / (2 * cp);
        const int v1 = imin(imax(L - r * cb, 0), cb);
        const int v2 = imin(imax(L - (2 * cp - 1 - r) * cb, 0), cb);
        acc += v1 + v2;
        acc1 += v1;
        acc2 += v2;
        if (p.cu_rank) p.cu_rank[r * (B + 1) + b + 1] = acc;
        if (p.cu_rank_half) {
          p.cu_rank_half[(r * 2 + 0) * (B + 1) + b + 1] = acc1;
          p.cu_rank_half[(r * 2 + 1) * (B + 1) + b + 1] = acc2;
        }
      }
      if (p.cu_rank_padded)
        for (int b = 0; b <= B; ++b) p.cu_rank_padded[r * (B + 1) + b] = PQ[b] / cp;
    }
  }
  if (p.token_map) {
    const int T = PQ[B];
    const int per = T / cp;
    for (int g = tid; g < T; g += nt) {
      const int b = upper_index(PQ, B, g);
      const int pos = g - PQ[b];
      const int cb = (PQ[b + 1] - PQ[b]) / (2 * cp);
      const int chunk = pos / cb;
      const int owner = chunk < cp ? chunk : 2 * cp - 1 - chunk;
      const int local = chunk == owner ? pos - owner * cb : cb + (pos - chunk * cb);
      p.token_map[owner * per + PQ[b] / cp + local] = g;
    }
  }
  if (p.mode == 0) return;
  const int32_t* effr = meta_in_smem ? s_meta : eff;
  if (!plan_schedule(p, effr, meta_in_smem ? s_meta + 4 * (B + 1) : p.tile_off, p.mode == 3 ? 2 : p.mode,
                     p.tile_off, p.counters, p.items, p.item_cap, s_warp, s_hist))
    return;
  if (p.mode == 3) {
    __syncthreads();  // s_hist and the staged tile offsets are reused
    plan_schedule(p, effr, meta_in_smem ? s_meta + 4 * (B + 1) : p.tile_off_q, 1, p.tile_off_q, p.counters_q,
                  p.items_q, p.item_cap_q, s_warp, s_hist);
  }
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t st) {
  prof_before(p.mode == 0 ? THD_KERNEL_PARTITION : THD_KERNEL_PLAN, st);
  plan_kernel<<<1, kPlanThreads, 0, st>>>(p);
  count_launch();
  cudaError_t e = cudaGetLastError();
  prof_after(p.mode == 0 ? THD_KERNEL_PARTITION : THD_KERNEL_PLAN, st);
  return e;
}

// ------------------------------------------------------------------ LSE merge
// (o_acc, lse_acc) <- merge with (o_part, lse_part).  A block owns a tile of
// tt consecutive tokens with all H heads: that tile's O rows are one
// contiguous stretch of memory, and for each head its lse values are tt
// contiguous floats.  Phase 1: each thread reads one (h, t) pair of lse
// values (coalesced), writes the merged lse back itself -- nothing else reads
// that entry, so there is no in-place race -- and leaves the two weights in
// shared memory.  Phase 2: the tile's O rows are streamed, one warp per row
// and kMergeRows rows per warp in flight, lanes over the row's float4s.
// PartT: float (fp32 partials) or uint16_t (bf16 partials, four per 8-byte
// load).
__device__ inline float4 load_part4(const float* p, int64_t i) { return __ldg(reinterpret_cast<const float4*>(p) + i); }
__device__ inline float4 load_part4(const uint16_t* p, int64_t i) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p) + i);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xffff0000u));
}

constexpr int kMergeRows = 4;          // O rows per warp in flight
constexpr int kMergeTileRows = 128;    // about H * tt rows per tile: many small tiles, so the
                                       // block scheduler balances the last wave

template <typename PartT>
__global__ void __launch_bounds__(256) lse_merge_kernel(float4* __restrict__ o_acc, float* __restrict__ lse_acc,
                                                        const PartT* __restrict__ o_part,
                                                        const float* __restrict__ lse_part, int64_t T, int H,
                                                        int D4, int tt) {
  extern __shared__ float s_w[];  // [2][H][tt]: the weights of the accumulator and of the partial
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const int64_t ntiles = (T + tt - 1) / tt;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t t0 = tile * tt;
    const int nt = (int)(T - t0 < tt ? T - t0 : tt);
    for (int i = threadIdx.x; i < H * nt; i += blockDim.x) {
      const int h = i / nt, tl = i - h * nt;
      const int64_t li = (int64_t)h * T + t0 + tl;
      const float a = lse_acc[li], b = __ldg(lse_part + li);
      const float hi = fmaxf(a, b), lo = fminf(a, b);
      float lse = -INFINITY, wa = 0.f, wb = 0.f;
      if (hi != -INFINITY) {  // a side at -inf contributes nothing; both -inf give (0, -inf)
        lse = hi + log1pf(expf(lo - hi));
        wa = a == -INFINITY ? 0.f : expf(a - lse);
        wb = b == -INFINITY ? 0.f : expf(b - lse);
      }
      lse_acc[li] = lse;
      s_w[h * tt + tl] = wa;
      s_w[(H + h) * tt + tl] = wb;
    }
    __syncthreads();
    const int nrows = nt * H;  // rows (t0 + tl) * H + h, in memory order
    const int64_t base = t0 * H * (int64_t)D4;
    for (int r0 = warp * kMergeRows; r0 < nrows; r0 += nwarp * kMergeRows) {
      float wa[kMergeRows], wb[kMergeRows];
#pragma unroll
      for (int u = 0; u < kMergeRows; ++u) {
        const int r = r0 + u;
        const int tl = r / H, h = r - tl * H;
        wa[u] = r < nrows ? s_w[h * tt + tl] : 0.f;
        wb[u] = r < nrows ? s_w[(H + h) * tt + tl] : 0.f;
      }
      for (int j = lane; j < D4; j += 32) {
        float4 x[kMergeRows], y[kMergeRows];
#pragma unroll
        for (int u = 0; u < kMergeRows; ++u)
          if (r0 + u < nrows) {
            x[u] = o_acc[base + (int64_t)(r0 + u) * D4 + j];
            y[u] = load_part4(o_part, base + (int64_t)(r0 + u) * D4 + j);
          }
#pragma unroll
        for (int u = 0; u < kMergeRows; ++u)
          if (r0 + u < nrows)
            o_acc[base + (int64_t)(r0 + u) * D4 + j] =
                make_float4(wa[u] * x[u].x + wb[u] * y[u].x, wa[u] * x[u].y + wb[u] * y[u].y,
                            wa[u] * x[u].z + wb[u] * y[u].z, wa[u] * x[u].w + wb[u] * y[u].w);
      }
    }
    __syncthreads();  // the weights are reused by the next tile
  }
}

template <typename PartT>
static cudaError_t launch_lse_merge_t(float* o_acc, float* lse_acc, const PartT* o_part, const float* lse_part,
                                      int64_t T, int H, int D, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int tt = H >= kMergeTileRows ? 1 : kMergeTileRows / H;
  const size_t smem = sizeof(float) * 2 * (size_t)H * tt;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(lse_merge_kernel<PartT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t ntiles = (T + tt - 1) / tt;
  const int grid = (int)(ntiles < (1LL << 20) ? ntiles : (1LL << 20));  // one tile per block
  prof_before(THD_KERNEL_LSE_MERGE, st);
  lse_merge_kernel<PartT><<<grid, 256, smem, st>>>((float4*)o_acc, lse_acc, o_part, lse_part, T, H, D / 4, tt);
  count_launch();
  cudaError_t e = cudaGetLastError();
  prof_after(THD_KERNEL_LSE_MERGE, st);
  return e;
}

cudaError_t launch_lse_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part, int64_t T,
                             int H, int D, cudaStream_t st) {
  return launch_lse_merge_t<float>(o_acc, lse_acc, o_part, lse_part, T, H, D, st);
}

cudaError_t launch_lse_merge_bf16(float* o_acc, float* lse_acc, const uint16_t* o_part, const float* lse_part,
                                  int64_t T, int H, int D, cudaStream_t st) {
  return launch_lse_merge_t<uint16_t>(o_acc, lse_acc, o_part, lse_part, T, H, D, st);
}

// ------------------------------------------------------------------ tail-zero
// Zero rows [*end, rows) of up to three [rows, H, D] bf16 buffers; reads the
// endpoint on the device, so it does nothing when there is no tail.
struct TailJob {
  uint16_t* buf;
  int64_t rows;
  int hd;  // H * D
  const int32_t* end;
};

__global__ void __launch_bounds__(256) tail_zero_kernel(TailJob j0, TailJob j1, TailJob j2,
                                                        const int32_t* dev_status) {
  if (dev_status && *dev_status != 0) return;
  TailJob jobs[3] = {j0, j1, j2};
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const TailJob& j = jobs[k];
    if (!j.buf) continue;
    // an endpoint outside [0, rows] is invalid metadata: nothing is written
    // (so a negative or oversized value can never move the writes outside
    // the buffer)
    const int64_t end = *j.end;
    if (end < 0 || end > j.rows) continue;
    const int64_t start = end * j.hd;
    const int64_t stop = j.rows * (int64_t)j.hd;
    // 16-byte stores (H * D is a multiple of 8)
    for (int64_t i = start + (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) * 8; i < stop;
         i += (int64_t)gridDim.x * blockDim.x * 8)
      *reinterpret_cast<uint4*>(j.buf + i) = make_uint4(0, 0, 0, 0);
  }
}

cudaError_t launch_tail_zero(uint16_t* dq, uint16_t* dk, uint16_t* dv, int64_t dq_rows, int64_t dkv_rows, int Hq,
                             int Hkv, int D, const int32_t* pad_q_end, const int32_t* pad_kv_end,
                             const int32_t* dev_status, cudaStream_t st) {
  TailJob a{dq, dq_rows, Hq * D, pad_q_end}, b{dk, dkv_rows, Hkv * D, pad_kv_end},
      c{dv, dkv_rows, Hkv * D, pad_kv_end};
  const int64_t biggest = (dq_rows * Hq > dkv_rows * Hkv ? dq_rows * Hq : dkv_rows * Hkv) * (int64_t)D / 8;
  const int64_t want = (biggest + 255) / 256;
  const int grid = (int)(want < 2LL * num_sms() ? (want > 0 ? want : 1) : 2LL * num_sms());
  prof_before(THD_KERNEL_TAIL_ZERO, st);
  tail_zero_kernel<<<grid, 256, 0, st>>>(a, b, c, dev_status);
  count_launch();
  cudaError_t e = cudaGetLastError();
  prof_after(THD_KERNEL_TAIL_ZERO, st);
  return e;
}

// ------------------------------------------------------------------ backward preprocess
// Delta[h][t] = sum_d dO[t,h,d] * O[t,h,d] and lse2[h][t] = lse * log2(e) on
// valid rows (0 elsewhere), read by both backward passes.
__device__ inline bool row_valid(const int32_t* eff, int B, int t) {
  const int32_t* cu = eff;
  const int32_t* pad = eff + (B + 1);
  if (t >= pad[B]) return false;
  const int b = upper_index(pad, B, t);
  return b < B && t - pad[b] < cu[b + 1] - cu[b];
}

// Sum of the eight bf16 x bf16 products of two 16-byte vectors, in fp32.
__device__ inline float dot8_bf16(const uint4& a, const uint4& b) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[k]));
    const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[k]));
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
  return acc;
}

// A CTA takes a tile of `tt` consecutive tokens with all Hq heads: those
// rows are one contiguous block of O and of dO, read with 16-byte loads, D/8
// lanes per row and kPrepBatch rows per thread in flight.  Delta is staged
// in shared memory as [Hq][tt], so Delta, lse and lse2 move as tt contiguous
// floats per head.
constexpr int kPrepThreads = 256;
constexpr int kPrepBatch = 4;
constexpr int kPrepMaxTok = 16;

template <int D>
__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                                const uint16_t* __restrict__ dout,
                                                                const float* __restrict__ lse,
                                                                float* __restrict__ delta, float* __restrict__ lse2,
                                                                const int32_t* __restrict__ eff, int B, int64_t T,
                                                                int Hq, int tt, const int32_t* dev_status) {
  extern __shared__ float s_delta[];  // [Hq][tt]
  __shared__ int s_valid[kPrepMaxTok];
  if (*dev_status != 0) return;
  constexpr int LPR = D / 8;                 // lanes per row
  constexpr int G = kPrepThreads / LPR;      // rows per pass
  const int tid = threadIdx.x, g = tid / LPR, j = tid % LPR;
  const int64_t ntiles = (T + tt - 1) / tt;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t t0 = tile * tt;
    const int nt = (int)(T - t0 < tt ? T - t0 : tt);
    if (tid < tt) s_valid[tid] = tid < nt && row_valid(eff, B, (int)(t0 + tid));
    __syncthreads();
    const int rows = nt * Hq;
    const uint4* po = reinterpret_cast<const uint4*>(o + t0 * Hq * D) + j;
    const uint4* pd = reinterpret_cast<const uint4*>(dout + t0 * Hq * D) + j;
    for (int r0 = 0; r0 < rows; r0 += G * kPrepBatch) {
      uint4 a[kPrepBatch], b[kPrepBatch];
#pragma unroll
      for (int u = 0; u < kPrepBatch; ++u) {
        const int r = r0 + u * G + g;
        a[u] = make_uint4(0, 0, 0, 0);
        b[u] = a[u];
        if (r < rows && s_valid[r / Hq]) {
          a[u] = __ldg(po + (int64_t)r * LPR);
          b[u] = __ldg(pd + (int64_t)r * LPR);
        }
      }
#pragma unroll
      for (int u = 0; u < kPrepBatch; ++u) {
        float acc = dot8_bf16(a[u], b[u]);
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const int r = r0 + u * G + g;
        if (j == 0 && r < rows) {
          const int tl = r / Hq;
          s_delta[(r - tl * Hq) * tt + tl] = acc;
        }
      }
    }
    __syncthreads();
    for (int i = tid; i < tt * Hq; i += kPrepThreads) {
      const int h = i / tt, tl = i - h * tt;
      if (tl < nt) {
        const int64_t gi = (int64_t)h * T + t0 + tl;
        delta[gi] = s_delta[i];
        // rows that see no key (bottom-right causal with L_q > L_kv) have
        // lse = -inf: 0 keeps their masked columns at 2^(-inf - 0) = 0
        // instead of -inf - (-inf)
        lse2[gi] = s_valid[tl] && lse[gi] != -INFINITY ? lse[gi] * 1.4426950408889634f : 0.f;
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_bwd_prep(const uint16_t* o, const uint16_t* dout, const float* lse, float* delta, float* lse2,
                            const int32_t* eff, int B, int64_t T_q, int Hq, int D, const int32_t* dev_status,
                            cudaStream_t st) {
  if (T_q == 0) return cudaSuccess;
  // tokens per tile: at most kPrepMaxTok, and the [Hq][tt] stage within 48 KB
  int tt = 12288 / Hq;
  tt = tt < 1 ? 1 : (tt > kPrepMaxTok ? kPrepMaxTok : tt);
  const size_t smem = sizeof(float) * (size_t)Hq * tt;
  const int64_t ntiles = (T_q + tt - 1) / tt;
  const int grid = (int)(ntiles < 8LL * num_sms() ? ntiles : 8LL * num_sms());
  auto kern = D == 128 ? bwd_prep_kernel<128> : bwd_prep_kernel<64>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  prof_before(THD_KERNEL_BWD_PREP, st);
  kern<<<grid, kPrepThreads, smem, st>>>(o, dout, lse, delta, lse2, eff, B, T_q, Hq, tt, dev_status);
  count_launch();
  cudaError_t e = cudaGetLastError();
  prof_after(THD_KERNEL_BWD_PREP, st);
  return e;
}

}  // namespace thd
