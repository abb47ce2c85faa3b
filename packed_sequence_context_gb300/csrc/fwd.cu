// Forward attention over packed THD tensors, decomposed like P2P (ring)
// context parallelism and executed for every emulated rank on one GB300.
//
// [P1] TransformerEngine issue #2208 (traceback through
// AttnFuncWithCPAndKVP2P.forward): per ring step, partial attention of the
// rank's local queries against the KV it holds, corrected into the running
// output.  [P3] "Hybrid / Hierarchical Context Parallel Skill" ("Contraintes
// requises"): sequences split into 2*cp chunks; rank r owns chunks r and
// 2cp-1-r.
//
// One work item = (rank r, sequence b, query head h, rank-local 128-row query
// tile t).  The item walks ring steps i = 0..cp-1 (KV of rank s = (r-i) mod
// cp: chunks s then 2cp-1-s) and, inside each, the 128-row key tiles that
// hold any key a query of the tile may see; fully masked tiles are skipped.
// The per-step LSE merge happens on chip: the running (max, sum, O) of the
// online softmax is exactly the log-sum-exp correction applied at tile
// granularity.  In one-step mode (thd_attn_fwd_step) only step `step_lo`
// is walked and the step's partial (O_i, lse_i) is written in fp32.
//
// CTA layout (384 threads, one CTA per SM, persistent over the schedule):
//   warps 0-7  softmax + epilogue in two warpgroups: a thread owns one query
//              row (its TMEM lane) and half of the key columns of each tile
//   warp 8     producer: gathers each item's query tile (its rows come from
//              two chunks, so cp.async row gathers) and issues the K tile TMA
//              loads (3-D tensor maps over [T, Hkv, D]) into a 3-slot ring
//   warp 10    producer of the V tiles (2-slot ring: a V slot frees only when
//              its PV completes, a K slot already when its QK^T does)
//   warp 9     TMEM allocator and QK^T issuer (one thread)
//   warp 11    PV issuer (one thread)
// TMEM: three S buffers of 128 fp32 columns ([0,384)); the softmax writes P
// as packed bf16 over the first columns of its S buffer, and PV reads it from
// TMEM as the A operand; O accumulates in [384, 384+D).  MMAs into different
// accumulators are not ordered among themselves, so a buffer is reused for a
// later QK^T only after the PV that read its P has completed (s_free).
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace thd {

template <int D>
struct FwdCfg {
  static constexpr int kKStages = D == 128 ? 3 : 4;  // K ring: a slot frees when its QK^T completes
  static constexpr int kVStages = D == 128 ? 2 : 3;  // V ring: a slot frees when its PV completes
  static constexpr int kQBytes = kTile * D * 2;
  static constexpr int kKVBytes = kTile * D * 2;  // one K (or V) tile
  static constexpr int kSmem = 1024 + kQBytes + (kKStages + kVStages) * kKVBytes;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kSBufs = 3;          // S/P buffers of 128 columns
  static constexpr uint32_t kColO = 384;
  static constexpr int kThreads = 384;
};

using FwdItem = QItem;

template <int D, bool kStep, bool kDyn>
__global__ void __launch_bounds__(384, 1)
    fwd_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = FwdCfg<D>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kQBytes;
  uint8_t* sV = sK + KS * C::kKVBytes;
  __shared__ __align__(8) uint64_t bar_k_full[KS];
  __shared__ __align__(8) uint64_t bar_k_empty[KS];
  __shared__ __align__(8) uint64_t bar_v_full[VS];
  __shared__ __align__(8) uint64_t bar_v_empty[VS];
  __shared__ __align__(8) uint64_t bar_s_full[C::kSBufs];
  __shared__ __align__(8) uint64_t bar_p_ready[C::kSBufs];
  __shared__ __align__(8) uint64_t bar_s_free[C::kSBufs];
  __shared__ __align__(8) uint64_t bar_q_full;
  __shared__ __align__(8) uint64_t bar_q_empty;
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ __align__(8) uint64_t bar_drain2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ ItemRing ring;             // items handed out to this CTA, in claim order
  __shared__ float s_mx[2][2][kTile];   // partial row maxima, [tile parity][half][row]
  __shared__ float s_sum[2][2][kTile];  // partial row sums, [item parity][half][row]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (*p.dev_status != 0) return;  // metadata rejected: outputs untouched
  const int n_entries = p.counters[0];
  const int n_items = n_entries * p.Hq;

  if (tid == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_k_empty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_v_empty[s], 1);
    }
    for (int s = 0; s < C::kSBufs; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_p_ready[s], 8);  // one arrival per softmax warp
      mbar_init(&bar_s_free[s], 1);
    }
    mbar_init(&bar_q_full, 32);
    mbar_init(&bar_q_empty, 1);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_drain2, 1);
    if constexpr (kDyn) item_ring_init(&ring, 3 + 8);  // warps 9, 10, 11 (one thread each) and the 8 softmax warps
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // Test hook (thd_test_arm_stall): every thread waits on a barrier nothing
  // completes, so the bounded wait runs out, the CTA takes the abort path
  // before any copy or MMA is issued, frees its TMEM and reports
  // THD_ERR_TIMEOUT.  The drain barrier is free for this: in this mode no
  // role runs, so nothing ever commits to it.
  if (p.test_stall) {
    mbar_wait(&bar_drain, 0, &s_abort);
  } else if (warp == 8) {
    // ------------------------------------------------------------ query + key producer (whole warp)
    int ks = 0;
    uint32_t kph = 0, n_fill = 0, q_iter = 0;
    bool ok = true;
    int w = item_first();
    for (uint32_t kit = 0; ok; ++kit) {
      int wnext = w + (int)gridDim.x;  // the fixed-stride walk
      if constexpr (kDyn) {
        // publish this item (or the end marker) to the other roles, and
        // claim the next one while this one is loaded
        if (lane == 0) {
          ok = item_publish(&ring, kit, w, &s_abort);
          if (ok && w < n_items) wnext = item_claim(p.claim);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      if (w >= n_items) break;
      const FwdItem it = q_item<kDyn>(p, n_entries, w);
      // ---- the query tile: rank-local rows [128 t, 128 t + 128) of rank r,
      // gathered into 128B-swizzled smem once the previous item's last QK^T
      // has completed; rows without a valid query are zero
      if (!mbar_wait(&bar_q_empty, (q_iter & 1u) ^ 1u, &s_abort)) break;
      const uint32_t qdst = smem_u32(sQ);
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int row = lane + 32 * rr;
        const int prow = it.t * kTile + row;
        const bool in_rank = prow < 2 * it.g.cbq;
        const int pos = in_rank ? local_to_pos(prow, it.r, it.g.cbq, p.cp) : 0;
        const bool valid = in_rank && pos < it.g.Lq;
        const uint16_t* src = valid ? p.q + (((int64_t)it.g.q_off + pos) * p.Hq + it.h) * D : p.q;
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
          cp_async_16(qdst + sw128_offset(row, 8 * c, kTile), src + (valid ? 8 * c : 0), valid ? 16u : 0u);
      }
      // the copies must have landed and be visible to the tensor core's
      // (async) proxy before the MMA thread may read them
      cp_async_wait_all();
      fence_proxy_async_smem();
      mbar_arrive(&bar_q_full);
      ++q_iter;
      // ---- the key tiles of the item, in ring order
      for_each_kv_tile(it, p, [&](int c, int j) {
        if (!ok) return;
        if (!mbar_wait(&bar_k_empty[ks], kph ^ 1u, &s_abort)) {
          ok = false;
          return;
        }
        if (lane == 0) {
          const int row = it.g.kv_off + c * it.g.cbkv + j * kTile;
          mbar_arrive_expect_tx(&bar_k_full[ks], C::kKVBytes);
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(smem_u32(sK + ks * C::kKVBytes + hb * 16384), &tmK, &bar_k_full[ks], hb * 64, it.kvh, row);
        }
        ++n_fill;
        if (++ks == KS) {
          ks = 0;
          kph ^= 1u;
        }
      });
      w = kDyn ? __shfl_sync(0xffffffffu, wnext, 0) : wnext;
    }
    // every issued load must land before the CTA may exit
    if (lane == 0) {
      for (int s = 0; s < KS; ++s) {
        const uint32_t fills = n_fill > (uint32_t)s ? (n_fill - 1 - s) / KS + 1 : 0;
        if (fills > 0) drain_wait(&bar_k_full[s], (fills - 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------ value producer
    if (lane == 0) {
      int vs = 0;
      uint32_t vph = 0, n_fill = 0;
      bool ok = true;
      for (uint32_t kit = 0; ok; ++kit) {
        int w = (int)(blockIdx.x + kit * gridDim.x);
        if constexpr (kDyn)
          if (!item_take_one(&ring, kit, w, &s_abort)) break;
        if (w >= n_items) break;
        const FwdItem it = q_item<kDyn>(p, n_entries, w);
        for_each_kv_tile(it, p, [&](int c, int j) {
          if (!ok) return;
          if (!mbar_wait(&bar_v_empty[vs], vph ^ 1u, &s_abort)) {
            ok = false;
            return;
          }
          const int row = it.g.kv_off + c * it.g.cbkv + j * kTile;
          mbar_arrive_expect_tx(&bar_v_full[vs], C::kKVBytes);
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(smem_u32(sV + vs * C::kKVBytes + hb * 16384), &tmV, &bar_v_full[vs], hb * 64, it.kvh, row);
          ++n_fill;
          if (++vs == VS) {
            vs = 0;
            vph ^= 1u;
          }
        });
      }
      for (int s = 0; s < VS; ++s) {
        const uint32_t fills = n_fill > (uint32_t)s ? (n_fill - 1 - s) / VS + 1 : 0;
        if (fills > 0) drain_wait(&bar_v_full[s], (fills - 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ QK^T issuer
    // The tensor pipe accepts an MMA only about as fast as it executes one,
    // so every barrier wait or commit in an issuing thread leaves it idle for
    // that long.  QK^T and PV are therefore issued by two threads (warps 9
    // and 11): while one waits on a barrier, the other keeps the pipe fed.
    // Ordering between the two streams comes only from the barriers: a QK^T
    // overwrites S buffer b once the PV that read P from it has completed
    // (s_free), and a PV reads P only after the softmax wrote it (p_ready).
    if (lane == 0) {
      const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kdesc = sdesc_sw128(smem_u32(sK), 16, 1024);
      int ks = 0;
      uint32_t kph = 0, g = 0, q_iter = 0;
      bool ok = true;
      for (uint32_t kit = 0; ok; ++kit) {
        int w = (int)(blockIdx.x + kit * gridDim.x);
        if constexpr (kDyn)
          if (!item_take_one(&ring, kit, w, &s_abort)) break;
        if (w >= n_items) break;
        const FwdItem it = q_item<kDyn>(p, n_entries, w);
        int n = 0;
        for_each_kv_tile(it, p, [&](int, int) { ++n; });
        if (!mbar_wait(&bar_q_full, q_iter & 1u, &s_abort)) break;
        ++q_iter;
        tc_fence_after();
        if (n == 0) tc_commit(&bar_q_empty);
        int j = 0;
        for_each_kv_tile(it, p, [&](int c, int jt) {
          if (!ok) return;
          const int ncols = q_tile_ncols(it, p, c, jt);
          const uint32_t b = g % C::kSBufs;
          if (!mbar_wait(&bar_k_full[ks], kph, &s_abort) ||
              (g >= (uint32_t)C::kSBufs && !mbar_wait(&bar_s_free[b], (g / C::kSBufs - 1) & 1u, &s_abort))) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint32_t idesc_qk = idesc_bf16(128, ncols, false, false);
          const uint64_t kd = kdesc + (uint64_t)((ks * C::kKVBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
            mma_ss(tmem + b * 128u, qdesc + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
          }
          tc_commit(&bar_s_full[b]);
          tc_commit(&bar_k_empty[ks]);                  // the K slot frees once this QK^T completes
          if (++j == n) tc_commit(&bar_q_empty);        // and the query tile after the item's last QK^T
          if (++ks == KS) {
            ks = 0;
            kph ^= 1u;
          }
          ++g;
        });
      }
      // all issued MMAs must complete before TMEM is released
      tc_commit(&bar_drain);
      drain_wait(&bar_drain, 0);
    }
    __syncwarp();
  } else if (warp == 11) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
      const uint64_t vdesc = sdesc_sw128(smem_u32(sV), 16384, 1024);
      int vs = 0;
      uint32_t vph = 0, g = 0;
      bool ok = true;
      for (uint32_t kit = 0; ok; ++kit) {
        int w = (int)(blockIdx.x + kit * gridDim.x);
        if constexpr (kDyn)
          if (!item_take_one(&ring, kit, w, &s_abort)) break;
        if (w >= n_items) break;
        const FwdItem it = q_item<kDyn>(p, n_entries, w);
        int j = 0;
        for_each_kv_tile(it, p, [&](int c, int jt) {
          if (!ok) return;
          const int ncols = q_tile_ncols(it, p, c, jt);
          const uint32_t b = g % C::kSBufs;
          if (!mbar_wait(&bar_p_ready[b], (g / C::kSBufs) & 1u, &s_abort) ||
              !mbar_wait(&bar_v_full[vs], vph, &s_abort)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint32_t pcol = tmem + b * 128u;
          const uint64_t vd = vdesc + (uint64_t)((vs * C::kKVBytes) >> 4);
          for (int kk = 0; kk < ncols / 16; ++kk)  // packed P of key columns 16 kk.. at 64 (kk/4) + 8 (kk%4)
            mma_ts(tmem + C::kColO, pcol + 64 * (kk >> 2) + 8 * (kk & 3), vd + (uint64_t)(kk * (2048 >> 4)), idesc_pv,
                   (j == 0 && kk == 0) ? 0u : 1u);
          tc_commit(&bar_v_empty[vs]);
          tc_commit(&bar_s_free[b]);  // PV on buffer b done: P consumed, O holds tile g
          if (++vs == VS) {
            vs = 0;
            vph ^= 1u;
          }
          ++g;
          ++j;
        });
      }
      tc_commit(&bar_drain2);
      drain_wait(&bar_drain2, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Two warpgroups: thread (half, row) owns query row `row` (its TMEM lane)
    // and key columns [64 half, 64 half + 64) of every tile, plus head-dim
    // columns [D/2 half, D/2 half + D/2) of O.  The two threads of a row swap
    // partial row maxima once per tile through shared memory (pair barrier)
    // and their partial row sums once per item.
    const int half = warp >> 2;
    const int row = tid & 127;
    const int pair_bar = 2 + (warp & 3);  // named barrier of warps w and w + 4
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    constexpr int DH = D / 2;
    const float sl2 = p.scale_log2;
    // O rows start at multiples of 128 bytes: 32-byte stores when O is 32-byte aligned
    const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
    uint32_t g = 0, n_item = 0;
    bool ok = true;
    for (uint32_t kit = 0; ok; ++kit) {
      int w = (int)(blockIdx.x + kit * gridDim.x);
      if constexpr (kDyn) {
        if (!item_take_warp(&ring, kit, w, &s_abort)) {
          ok = false;
          break;
        }
      }
      if (w >= n_items) break;
      const FwdItem it = q_item<kDyn>(p, n_entries, w);
      const int prow = it.t * kTile + row;
      const bool in_rank = prow < 2 * it.g.cbq;
      const int pos = in_rank ? local_to_pos(prow, it.r, it.g.cbq, p.cp) : 0;
      const bool valid = in_rank && pos < it.g.Lq;
      const int64_t grow = (int64_t)it.g.q_off + pos;
      // ---- key tiles
      float m = -INFINITY, l = 0.f;  // running max (log2 units, shared value) and this half's sum
      int jl = 0;
      for_each_kv_tile(it, p, [&](int c, int j) {
        if (!ok) return;
        const uint32_t sb = g % C::kSBufs;
        if (!mbar_wait(&bar_s_full[sb], (g / C::kSBufs) & 1u, &s_abort)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const int j0 = c * it.g.cbkv + j * kTile;
        int cnt = 0;
        if (valid) {
          cnt = imin(kTile, (c + 1) * it.g.cbkv - j0);
          cnt = imin(cnt, it.g.Lkv - j0);
          if (p.causal) cnt = imin(cnt, pos + it.g.koff - j0 + 1);
          cnt = imax(cnt, 0);
        }
        const int ncols = q_tile_ncols(it, p, c, j);  // the N this tile's QK^T computed
        const int nch = ceil_div(ncols, 32);
        const int k0 = 2 * half;  // this thread's 32-column chunks: k0, k0 + 1
        uint32_t sr[2][32];
        const uint32_t scol = tmem + lane_base + sb * 128u;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          if (k0 + kk < nch) tmem_ld32(scol + 32 * (k0 + kk), sr[kk]);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          if (k0 + kk < nch) tmem_ld_wait(sr[kk]);
        // keys past the row's last visible one count as -inf; whole warps of
        // fully visible rows (every tile off the causal diagonal) skip the selects
        const int nvalid = (k0 + 1 < nch) ? 64 : (k0 < nch ? 32 : 0);  // this thread's loaded columns
        if (__any_sync(0xffffffffu, cnt - 32 * k0 < nvalid)) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int n = 0; n < 32; ++n)
              if (32 * (k0 + kk) + n >= cnt) sr[kk][n] = __float_as_uint(-INFINITY);
        }
        if (k0 + 1 >= nch) {  // chunks this thread did not load (narrow tile)
#pragma unroll
          for (int n = 0; n < 32; ++n) sr[1][n] = __float_as_uint(-INFINITY);
          if (k0 >= nch) {
#pragma unroll
            for (int n = 0; n < 32; ++n) sr[0][n] = __float_as_uint(-INFINITY);
          }
        }
        // tree maximum: eight independent partial maxima of 8 values each
        float pm[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t* v = &sr[i >> 2][8 * (i & 3)];
          float a = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
          a = fmax3(a, __uint_as_float(v[3]), __uint_as_float(v[4]));
          a = fmax3(a, __uint_as_float(v[5]), __uint_as_float(v[6]));
          pm[i] = fmaxf(a, __uint_as_float(v[7]));
        }
        const float mloc = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
        s_mx[g & 1u][half][row] = mloc;
        named_bar_sync(pair_bar, 64);
        const float mt = fmaxf(mloc, s_mx[g & 1u][half ^ 1][row]) * sl2;
        // lazy rescale: move the running max only when it grows by > 8 (log2 units)
        const bool upd = mt > m + 8.0f;
        const float alpha = upd ? ex2(m - mt) : 1.0f;
        const bool need_o = upd && (m != -INFINITY) && (jl > 0);
        if (upd) {
          l *= alpha;
          m = mt;
        }
        if (__any_sync(0xffffffffu, need_o)) {
          // O must hold the previous tile's PV before it is rescaled.  Its
          // buffer's s_free barrier is at most one phase behind (the PV before
          // it on that buffer completed before this item's QK reused it), so a
          // parity wait is exact there; a single barrier for all PVs is not.
          if (!mbar_wait(&bar_s_free[(g - 1) % C::kSBufs], ((g - 1) / C::kSBufs) & 1u, &s_abort)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const float f = need_o ? alpha : 1.0f;
#pragma unroll 1
          for (int k = 0; k < DH / 32; ++k) {
            uint32_t o[32];
            const uint32_t oc = tmem + lane_base + C::kColO + half * DH + 32 * k;
            tmem_ld32(oc, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int n = 0; n < 32; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * f);
            tmem_st32(oc, o);
          }
        }
        const float mm = (m == -INFINITY) ? 0.f : m;
        // P = 2^(S scale_log2 - m): the scale-and-shift as packed pair FMAs,
        // the row sum in four packed accumulators (short dependency chains)
        float sa[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          if (k0 + kk < nch) {
            uint32_t pk[16];
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(sr[kk][2 * n]), __uint_as_float(sr[kk][2 * n + 1]), sl2, sl2, -mm, -mm);
              const float p0 = ex2(x0), p1 = ex2(x1);
              const int a = 2 * (n & 3);
              fadd2(sa[a], sa[a + 1], sa[a], sa[a + 1], p0, p1);
              pk[n] = pack_bf16x2(p0, p1);
            }
            // packed P stays inside this half's own S columns (the partner may
            // still be reading its half): chunk k -> column 64 (k/2) + 16 (k%2)
            tmem_st16(scol + 64 * half + 16 * kk, pk);
          }
        }
        fadd2(sa[0], sa[1], sa[0], sa[1], sa[2], sa[3]);
        fadd2(sa[4], sa[5], sa[4], sa[5], sa[6], sa[7]);
        fadd2(sa[0], sa[1], sa[0], sa[1], sa[4], sa[5]);
        const float rs = sa[0] + sa[1];
        l += rs;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();  // every lane's P is in TMEM: one arrival speaks for the warp
        if (lane == 0) mbar_arrive(&bar_p_ready[sb]);
        ++g;
        ++jl;
      });
      if (!ok) break;
      // ---- epilogue
      if (jl > 0) {  // the last PV (and, in order, every earlier one) has completed
        if (!mbar_wait(&bar_s_free[(g - 1) % C::kSBufs], ((g - 1) / C::kSBufs) & 1u, &s_abort)) break;
        tc_fence_after();
      }
      s_sum[n_item & 1u][half][row] = l;
      named_bar_sync(pair_bar, 64);
      const float ltot = l + s_sum[n_item & 1u][half ^ 1][row];
      ++n_item;
      const bool live = valid && ltot > 0.f;
      const float inv_l = live ? 1.0f / ltot : 0.f;
      if (in_rank && half == 0) {
        const float lse = live ? (m + log2f(ltot)) * 0.69314718055994531f : -INFINITY;
        p.lse[(int64_t)it.h * p.T_q + grow] = lse;
      }
#pragma unroll 1
      for (int k = 0; k < DH / 32; ++k) {
        uint32_t o[32];
        if (jl > 0) {
          tmem_ld32(tmem + lane_base + C::kColO + half * DH + 32 * k, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int n = 0; n < 32; ++n) o[n] = 0u;
        }
        if (in_rank) {
          const int64_t col = (grow * p.Hq + it.h) * D + half * DH + 32 * k;
          if constexpr (kStep)
            store32_f32(static_cast<float*>(p.o) + col, o, inv_l, o_v8);
          else
            store32_bf16(static_cast<uint16_t*>(p.o) + col, o, inv_l, o_v8);
        }
      }
      tc_fence_before();
    }
    // ---- rows past the last sequence: O = 0, lse = -inf
    if (ok) {
      const int Tend = p.eff[(p.B + 1) + p.B];
      const int64_t nrow = (p.T_q - Tend) * (int64_t)p.Hq;
      for (int64_t i = (int64_t)blockIdx.x * 256 + tid; i < nrow; i += (int64_t)gridDim.x * 256) {
        const int64_t t = Tend + i / p.Hq;
        const int h = (int)(i % p.Hq);
        if constexpr (kStep) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + (t * p.Hq + h) * D);
          for (int n = 0; n < D / 4; ++n) dst[n] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + (t * p.Hq + h) * D);
          for (int n = 0; n < D / 8; ++n) dst[n] = make_uint4(0, 0, 0, 0);
        }
        p.lse[(int64_t)h * p.T_q + t] = -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && s_abort) atomicCAS(p.dev_status, 0, THD_ERR_TIMEOUT);
}

template <int D, bool kStep, bool kDyn>
static cudaError_t launch_fwd_t(const FwdParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                cudaStream_t st) {
  using C = FwdCfg<D>;
  cudaError_t ea =
      cudaFuncSetAttribute(fwd_kernel<D, kStep, kDyn>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (ea != cudaSuccess) return ea;
  prof_before(THD_KERNEL_FWD, st);
  fwd_kernel<D, kStep, kDyn><<<grid, C::kThreads, C::kSmem, st>>>(p, tk, tv);
  count_launch();
  cudaError_t e = cudaGetLastError();
  prof_after(THD_KERNEL_FWD, st);
  return e;
}

template <int D>
static cudaError_t launch_fwd_d(const FwdParams& p, const CUtensorMap& tk, const CUtensorMap& tv, bool step_mode,
                                bool dyn, int grid, cudaStream_t st) {
  if (step_mode)
    return dyn ? launch_fwd_t<D, true, true>(p, tk, tv, grid, st) : launch_fwd_t<D, true, false>(p, tk, tv, grid, st);
  return dyn ? launch_fwd_t<D, false, true>(p, tk, tv, grid, st) : launch_fwd_t<D, false, false>(p, tk, tv, grid, st);
}

cudaError_t launch_fwd(const FwdParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int D, bool step_mode,
                       bool dyn, int grid, cudaStream_t st) {
  return D == 128 ? launch_fwd_d<128>(p, tk, tv, step_mode, dyn, grid, st)
                  : launch_fwd_d<64>(p, tk, tv, step_mode, dyn, grid, st);
}

}  // namespace thd
