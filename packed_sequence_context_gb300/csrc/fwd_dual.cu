// Forward attention over packed THD tensors, decomposed like P2P (ring)
// context parallelism: the kernel for sequences of up to a few thousand
// tokens (short work items), with two items in flight per CTA.
//
// [P1] TransformerEngine issue #2208 (traceback through
// AttnFuncWithCPAndKVP2P.forward): per ring step, partial attention of the
// rank's local queries against the KV it holds, corrected into the running
// output.  [P3] "Hybrid / Hierarchical Context Parallel Skill" ("Contraintes
// requises"): sequences split into 2*cp chunks; rank r owns chunks r and
// 2cp-1-r.
//
// Work items, the ring walk and the on-chip LSE merge are those of the
// single-item forward kernel (fwd.cu): item = (rank r, sequence b, query
// head h, rank-local 128-row query tile t), walking ring steps i = 0..cp-1
// (KV of rank s = (r-i) mod cp: chunks s then 2cp-1-s) and the key tiles any
// query of the tile may see; one-step mode writes step `step_lo`'s partial.
//
// Two items in flight.  The CTA runs two independent streams of work items;
// each stream has its own query buffer, key and value slots, S and O
// accumulators in TMEM, producer warp, MMA-issuing thread and softmax
// warpgroup.  Inside a stream a key tile's steps are serial (S = QK^T, the
// softmax, O += PV, then the next S into the same TMEM columns); across the
// streams they overlap, so while one warpgroup runs the softmax of its tile
// the tensor pipe runs the other stream's products, and one stream's item
// changes (query gather, output stores, the wait for the next item's first
// S) hide behind the other's tiles.  A thread owns one whole query row, so
// no per-tile exchange between threads is needed.  On batches of sequences
// of 0.1-8K tokens (items of 1-30 key tiles) this measured 3-13% faster than
// the single-item kernel; on long sequences, where the single-item kernel's
// three S buffers keep the tensor pipe busy through the softmax, 15% slower.
//
// CTA layout (384 threads, one CTA per SM, persistent over the schedule):
//   warps 0-3, 4-7  softmax + epilogue of stream 0, 1 (thread = query row =
//                   its TMEM lane, every key column of its tiles)
//   warps 8, 9      producers of stream 0, 1: the query tile (its rows come
//                   from two chunks, so cp.async row gathers into 128B-swizzled
//                   smem) and the K and V tiles (TMA, 3-D tensor maps over
//                   [T, Hkv, D])
//   warps 10, 11    MMA issuers of stream 0, 1 (one thread each); warp 10 also
//                   allocates TMEM
// TMEM (512 columns): S of stream x in [128x, 128x + 128), P written back over
// its first 64 columns as packed bf16 (PV reads it from TMEM as the A
// operand); O of stream x in [256 + 128x, 256 + 128x + D).
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace thd {

template <int D>
struct FwdDualCfg {
  // key and value slots per stream: a K slot frees when its QK^T completes,
  // a V slot when its PV completes
  static constexpr int kKStages = D == 128 ? 1 : 2;
  static constexpr int kVStages = D == 128 ? 1 : 2;
  static constexpr int kQBytes = kTile * D * 2;
  static constexpr int kKVBytes = kTile * D * 2;  // one K (or V) tile
  static constexpr int kStreamBytes = kQBytes + (kKStages + kVStages) * kKVBytes;
  static constexpr int kSmem = 1024 + 2 * kStreamBytes;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kSoftmaxRegs = 200;  // per thread, warps 0-7
  static constexpr uint32_t kOtherRegs = 96;      // per thread, warps 8-11
  static_assert(256 * kSoftmaxRegs + 128 * kOtherRegs <= 384 * 168, "register split above the launch budget");
};

// Barriers of one stream.
struct FwdStreamBars {
  uint64_t k_full[2], k_empty[2];  // K slots (up to two)
  uint64_t v_full[2], v_empty[2];  // V slots
  uint64_t q_full;                 // query tile gathered (32 producer lanes)
  uint64_t q_empty;                // the item's last QK^T completed
  uint64_t s_full;                 // QK^T completed: S in TMEM
  uint64_t p_ready;                // P in TMEM (one arrival per softmax warp)
  uint64_t s_free;                 // PV completed: P consumed, O updated
  uint64_t drain;                  // the issuer's MMAs all completed
};

// Work items are handed out dynamically: every stream starts with item
// blockIdx.x + x gridDim.x, then its producer claims the next free item from
// the per-launch counter (items 2 gridDim.x and up) and publishes it to the
// stream's other roles through the stream's item ring.  The item map puts
// groups of kv heads outermost (with one group it is entry-major, every
// query head of a schedule entry side by side).
__device__ inline int fwd_dual_first_item(int x) { return (int)blockIdx.x + x * (int)gridDim.x; }

template <int D, bool kStep>
__global__ void __launch_bounds__(384, 1)
    fwd_dual_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = FwdDualCfg<D>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) FwdStreamBars bars[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ ItemRing ring[2];  // items handed out to each stream, in claim order

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (*p.dev_status != 0) return;  // metadata rejected: outputs untouched
  const int n_entries = p.counters[0];
  const int n_items = n_entries * p.Hq;

  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      FwdStreamBars& b = bars[x];
      for (int s = 0; s < KS; ++s) {
        mbar_init(&b.k_full[s], 1);
        mbar_init(&b.k_empty[s], 1);
      }
      for (int s = 0; s < VS; ++s) {
        mbar_init(&b.v_full[s], 1);
        mbar_init(&b.v_empty[s], 1);
      }
      mbar_init(&b.q_full, 32);
      mbar_init(&b.q_empty, 1);
      mbar_init(&b.s_full, 1);
      mbar_init(&b.p_ready, 4);  // one arrival per softmax warp of the stream
      mbar_init(&b.s_free, 1);
      mbar_init(&b.drain, 1);
      item_ring_init(&ring[x], 1 + 4);  // the issuer and the 4 softmax warps
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 10) {
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
  // THD_ERR_TIMEOUT.  Stream 0's drain barrier is free for this: in this mode
  // no role runs, so nothing ever commits to it.
  if (p.test_stall) {
    mbar_wait(&bars[0].drain, 0, &s_abort);
  } else if (warp >= 8) {
    // Registers: the softmax warpgroups hold a whole row of S (128 values)
    // per thread, the producer and issuer warps need few.  Each warpgroup
    // changes its budget at the top of its role (one instruction for all its
    // warps); 256 x kSoftmaxRegs + 128 x kOtherRegs fits the 384 x 168 the
    // CTA is launched with.
    regs_lower<C::kOtherRegs>();
    if (warp < 10) {
      // ------------------------------------------------------------ producer of stream x (whole warp)
      const int x = warp - 8;
      FwdStreamBars& sb = bars[x];
      uint8_t* sQ = smem + x * C::kStreamBytes;
      uint8_t* sK = sQ + C::kQBytes;
      uint8_t* sV = sK + KS * C::kKVBytes;
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0, nk = 0, nv = 0, q_iter = 0;
      bool ok = true;
      int w = fwd_dual_first_item(x);
      for (uint32_t kit = 0; ok; ++kit) {
        // publish this item (or the end marker) to the stream's other roles,
        // and claim the next one while this one is loaded
        int wnext = 0;
        if (lane == 0) {
          ok = item_publish(&ring[x], kit, w, &s_abort);
          if (ok && w < n_items) wnext = 2 * (int)gridDim.x + atomicAdd(p.claim, 1);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (w >= n_items) break;
        const QItem it = q_item<true>(p, n_entries, w);
        // ---- the query tile: rank-local rows [128 t, 128 t + 128) of rank r,
        // gathered once the previous item's last QK^T has completed; rows
        // without a valid query are zero.  The copies are waited for after the
        // item's first K load has been issued, so the two latencies overlap.
        if (!mbar_wait(&sb.q_empty, (q_iter & 1u) ^ 1u, &s_abort)) break;
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
        bool q_pending = true;
        // the copies must have landed and be visible to the tensor core's
        // (async) proxy before the MMA thread may read them
        auto finish_q = [&]() {
          cp_async_wait_all();
          fence_proxy_async_smem();
          mbar_arrive(&sb.q_full);
          q_pending = false;
        };
        // ---- the key and value tiles of the item, in ring order
        for_each_kv_tile(it, p, [&](int c, int j) {
          if (!ok) return;
          const int row = it.g.kv_off + c * it.g.cbkv + j * kTile;
          if (!mbar_wait(&sb.k_empty[ks], kph ^ 1u, &s_abort)) {
            ok = false;
            return;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&sb.k_full[ks], C::kKVBytes);
#pragma unroll
            for (int hb = 0; hb < D / 64; ++hb)
              tma_load_3d(smem_u32(sK + ks * C::kKVBytes + hb * 16384), &tmK, &sb.k_full[ks], hb * 64, it.kvh, row);
          }
          ++nk;
          if (++ks == KS) {
            ks = 0;
            kph ^= 1u;
          }
          if (q_pending) finish_q();
          if (!mbar_wait(&sb.v_empty[vs], vph ^ 1u, &s_abort)) {
            ok = false;
            return;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&sb.v_full[vs], C::kKVBytes);
#pragma unroll
            for (int hb = 0; hb < D / 64; ++hb)
              tma_load_3d(smem_u32(sV + vs * C::kKVBytes + hb * 16384), &tmV, &sb.v_full[vs], hb * 64, it.kvh, row);
          }
          ++nv;
          if (++vs == VS) {
            vs = 0;
            vph ^= 1u;
          }
        });
        if (!ok) break;
        if (q_pending) finish_q();  // an item without key tiles
        ++q_iter;
        w = __shfl_sync(0xffffffffu, wnext, 0);
      }
      // every issued copy must land before the CTA may exit
      cp_async_wait_all();
      if (lane == 0) {
        for (int s = 0; s < KS; ++s) {
          const uint32_t fills = nk > (uint32_t)s ? (nk - 1 - s) / KS + 1 : 0;
          if (fills > 0) drain_wait(&sb.k_full[s], (fills - 1) & 1u);
        }
        for (int s = 0; s < VS; ++s) {
          const uint32_t fills = nv > (uint32_t)s ? (nv - 1 - s) / VS + 1 : 0;
          if (fills > 0) drain_wait(&sb.v_full[s], (fills - 1) & 1u);
        }
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ MMA issuer of stream x
      // Per key tile: S = QK^T once the tile's K has landed, then O += PV once
      // the softmax has written P and the tile's V has landed.  While this
      // thread waits, the other stream's issuer keeps the pipe fed.
      const int x = warp - 10;
      FwdStreamBars& sb = bars[x];
      uint8_t* sQ = smem + x * C::kStreamBytes;
      uint8_t* sK = sQ + C::kQBytes;
      uint8_t* sV = sK + KS * C::kKVBytes;
      if (lane == 0) {
        const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t kdesc = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t vdesc = sdesc_sw128(smem_u32(sV), 16384, 1024);
        const uint32_t s_col = tmem + 128u * (uint32_t)x;
        const uint32_t o_col = tmem + C::kColO + 128u * (uint32_t)x;
        constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
        int ks = 0, vs = 0;
        uint32_t kph = 0, vph = 0, g = 0, q_iter = 0;
        bool ok = true;
        for (uint32_t kit = 0; ok; ++kit) {
          int w = 0;
          if (!item_take_one(&ring[x], kit, w, &s_abort)) break;
          if (w >= n_items) break;
          const QItem it = q_item<true>(p, n_entries, w);
          int n = 0;
          for_each_kv_tile(it, p, [&](int, int) { ++n; });
          if (!mbar_wait(&sb.q_full, q_iter & 1u, &s_abort)) break;
          ++q_iter;
          tc_fence_after();
          if (n == 0) tc_commit(&sb.q_empty);
          int j = 0;
          for_each_kv_tile(it, p, [&](int c, int jt) {
            if (!ok) return;
            const int ncols = q_tile_ncols(it, p, c, jt);
            // S of this tile overwrites the P the previous PV reads: both are
            // issued by this thread, and the tensor pipe executes one thread's
            // MMAs in issue order, so no wait for that PV is needed here
            if (!mbar_wait(&sb.k_full[ks], kph, &s_abort)) {
              ok = false;
              return;
            }
            tc_fence_after();
            const uint32_t idesc_qk = idesc_bf16(128, ncols, false, false);
            const uint64_t kd = kdesc + (uint64_t)((ks * C::kKVBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
              mma_ss(s_col, qdesc + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
            }
            tc_commit(&sb.s_full);
            tc_commit(&sb.k_empty[ks]);                // the K slot frees once this QK^T completes
            if (j + 1 == n) tc_commit(&sb.q_empty);    // and the query tile after the item's last QK^T
            if (++ks == KS) {
              ks = 0;
              kph ^= 1u;
            }
            if (!mbar_wait_poll(&sb.p_ready, g & 1u, &s_abort) || !mbar_wait(&sb.v_full[vs], vph, &s_abort)) {
              ok = false;
              return;
            }
            tc_fence_after();
            const uint64_t vd = vdesc + (uint64_t)((vs * C::kKVBytes) >> 4);
            // packed P of key columns [16 kk, 16 kk + 16) sits in TMEM columns [8 kk, 8 kk + 8)
            for (int kk = 0; kk < ncols / 16; ++kk)
              mma_ts(o_col, s_col + 8u * (uint32_t)kk, vd + (uint64_t)(kk * (2048 >> 4)), idesc_pv,
                     (j == 0 && kk == 0) ? 0u : 1u);
            tc_commit(&sb.v_empty[vs]);
            tc_commit(&sb.s_free);  // P consumed, O holds this tile
            if (++vs == VS) {
              vs = 0;
              vph ^= 1u;
            }
            ++g;
            ++j;
          });
        }
        // all issued MMAs must complete before TMEM is released
        tc_commit(&sb.drain);
        drain_wait(&sb.drain, 0);
      }
      __syncwarp();
    }
  } else {
    regs_raise<C::kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax + epilogue of stream x
    // Thread = query row `row` of the stream's items (TMEM lane), all key
    // columns of each tile and all D columns of O.
    const int x = warp >> 2;
    FwdStreamBars& sb = bars[x];
    const int row = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + 128u * (uint32_t)x;
    const uint32_t o_col = tmem + lane_base + C::kColO + 128u * (uint32_t)x;
    const float sl2 = p.scale_log2;
    // O rows start at multiples of 128 bytes: 32-byte stores when O is 32-byte aligned
    const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t kit = 0; ok; ++kit) {
      int w = 0;
      if (!item_take_warp(&ring[x], kit, w, &s_abort)) {
        ok = false;
        break;
      }
      if (w >= n_items) break;
      const QItem it = q_item<true>(p, n_entries, w);
      const int prow = it.t * kTile + row;
      const bool in_rank = prow < 2 * it.g.cbq;
      const int pos = in_rank ? local_to_pos(prow, it.r, it.g.cbq, p.cp) : 0;
      const bool valid = in_rank && pos < it.g.Lq;
      const int64_t grow = (int64_t)it.g.q_off + pos;
      // ---- key tiles
      float m = -INFINITY, l = 0.f;  // running max (log2 units) and sum of the row
      int jl = 0;
      for_each_kv_tile(it, p, [&](int c, int j) {
        if (!ok) return;
        if (!mbar_wait(&sb.s_full, g & 1u, &s_abort)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const int j0 = c * it.g.cbkv + j * kTile;
        int cnt = 0;  // keys of the tile this row sees
        if (valid) {
          cnt = imin(kTile, (c + 1) * it.g.cbkv - j0);
          cnt = imin(cnt, it.g.Lkv - j0);
          if (p.causal) cnt = imin(cnt, pos + it.g.koff - j0 + 1);
          cnt = imax(cnt, 0);
        }
        const int ncols = q_tile_ncols(it, p, c, j);  // the N this tile's QK^T computed
        const int nch = ceil_div(ncols, 32);          // 32-column chunks holding S
        uint32_t sr[4][32];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k < nch) tmem_ld32(s_col + 32 * k, sr[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k < nch) tmem_ld_wait(sr[k]);
        // keys past the row's last visible one count as -inf; whole warps of
        // fully visible rows (every tile off the causal diagonal) skip the selects
        if (__any_sync(0xffffffffu, cnt < 32 * nch)) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int n = 0; n < 32; ++n)
              if (32 * k + n >= cnt) sr[k][n] = __float_as_uint(-INFINITY);
        }
        // row maximum: per chunk four independent partial maxima of 8 values
        float mloc = -INFINITY;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (k < nch) {
            float pm[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t* v = &sr[k][8 * i];
              pm[i] = fmax3(fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2])),
                            fmax3(__uint_as_float(v[3]), __uint_as_float(v[4]), __uint_as_float(v[5])),
                            fmaxf(__uint_as_float(v[6]), __uint_as_float(v[7])));
            }
            mloc = fmax3(mloc, fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
          }
        }
        const float mt = mloc * sl2;
        // lazy rescale: move the running max only when it grows by > 8 (log2 units)
        const bool upd = mt > m + 8.0f;
        const float alpha = upd ? ex2(m - mt) : 1.0f;
        const bool need_o = upd && (m != -INFINITY) && (jl > 0);
        if (upd) {
          l *= alpha;
          m = mt;
        }
        if (__any_sync(0xffffffffu, need_o)) {
          // O holds the previous tile's PV: this tile's QK^T was issued only
          // after it completed.  The wait on its s_free phase is exact (the
          // next phase needs this warpgroup's P) and returns at once; it
          // orders the TMEM accesses below after that PV.
          if (!mbar_wait(&sb.s_free, (g - 1) & 1u, &s_abort)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const float f = need_o ? alpha : 1.0f;
#pragma unroll 1
          for (int k = 0; k < D / 32; ++k) {
            uint32_t o[32];
            tmem_ld32(o_col + 32 * k, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int n = 0; n < 32; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * f);
            tmem_st32(o_col + 32 * k, o);
          }
        }
        const float mm = (m == -INFINITY) ? 0.f : m;
        // P = 2^(S scale_log2 - m): the scale-and-shift as packed pair FMAs,
        // the row sum in four packed accumulators (short dependency chains);
        // packed P of key columns [32 k, 32 k + 32) goes to TMEM columns
        // [16 k, 16 k + 16), all of which this thread has already read
        float sa[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (k < nch) {
            uint32_t pk[16];
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(sr[k][2 * n]), __uint_as_float(sr[k][2 * n + 1]), sl2, sl2, -mm, -mm);
              const float p0 = ex2(x0), p1 = ex2(x1);
              const int a = 2 * (n & 3);
              fadd2(sa[a], sa[a + 1], sa[a], sa[a + 1], p0, p1);
              pk[n] = pack_bf16x2(p0, p1);
            }
            tmem_st16(s_col + 16 * k, pk);
          }
        }
        fadd2(sa[0], sa[1], sa[0], sa[1], sa[2], sa[3]);
        fadd2(sa[4], sa[5], sa[4], sa[5], sa[6], sa[7]);
        fadd2(sa[0], sa[1], sa[0], sa[1], sa[4], sa[5]);
        l += sa[0] + sa[1];
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();  // every lane's P is in TMEM: one arrival speaks for the warp
        if (lane == 0) mbar_arrive(&sb.p_ready);
        ++g;
        ++jl;
      });
      if (!ok) break;
      // ---- epilogue
      if (jl > 0) {  // the last PV (and, in order, every earlier one) has completed
        if (!mbar_wait(&sb.s_free, (g - 1) & 1u, &s_abort)) break;
        tc_fence_after();
      }
      const bool live = valid && l > 0.f;
      const float inv_l = live ? 1.0f / l : 0.f;
      if (in_rank) {
        const float lse = live ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[(int64_t)it.h * p.T_q + grow] = lse;
      }
#pragma unroll 1
      for (int k = 0; k < D / 32; ++k) {
        uint32_t o[32];
        if (jl > 0) {
          tmem_ld32(o_col + 32 * k, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int n = 0; n < 32; ++n) o[n] = 0u;
        }
        if (in_rank) {
          const int64_t col = (grow * p.Hq + it.h) * D + 32 * k;
          if constexpr (kStep)
            store32_f32(static_cast<float*>(p.o) + col, o, inv_l, o_v8);
          else
            store32_bf16(static_cast<uint16_t*>(p.o) + col, o, inv_l, o_v8);
        }
      }
      // the next item's first PV overwrites O: its p_ready arrival, after
      // these loads, orders them before it
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
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && s_abort) atomicCAS(p.dev_status, 0, THD_ERR_TIMEOUT);
}
template <int D, bool kStep>
static cudaError_t launch_fwd_dual_t(const FwdParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                     cudaStream_t st) {
  using C = FwdDualCfg<D>;
  cudaError_t ea =
      cudaFuncSetAttribute(fwd_dual_kernel<D, kStep>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (ea != cudaSuccess) return ea;
  prof_before(THD_KERNEL_FWD, st);
  fwd_dual_kernel<D, kStep><<<grid, C::kThreads, C::kSmem, st>>>(p, tk, tv);
  count_launch();
  cudaError_t e = cudaGetLastError();
  prof_after(THD_KERNEL_FWD, st);
  return e;
}

cudaError_t launch_fwd_dual(const FwdParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int D, bool step_mode,
                            int grid, cudaStream_t st) {
  if (D == 128) return step_mode ? launch_fwd_dual_t<128, true>(p, tk, tv, grid, st)
                                 : launch_fwd_dual_t<128, false>(p, tk, tv, grid, st);
  return step_mode ? launch_fwd_dual_t<64, true>(p, tk, tv, grid, st) : launch_fwd_dual_t<64, false>(p, tk, tv, grid, st);
}

}  // namespace thd
