// dQ of attention over packed THD tensors, query-stationary, walked in the
// same P2P ring order as the forward and executed for every emulated rank on
// one GB300.
//
// [P2] TransformerEngine issue #3487 ("Steps/Code to reproduce bug": BF16
// attention backward on this layout with four-rank P2P context parallelism;
// "Describe the bug": THD dQ tail-zeroing).  [P1] TransformerEngine issue
// #2208 (traceback through AttnFuncWithCPAndKVP2P): at ring step i rank r
// holds the KV of rank s = (r - i) mod cp and accumulates its dQ partial from
// it.  The key/value-stationary kernel produces dK and dV; this one recomputes
// S and dP for its own query tile and keeps dQ on chip for the whole walk, so
// dQ needs no atomics and no fp32 accumulator in global memory.
//
// One work item = (rank r, sequence b, query head h, rank-local 128-row query
// tile t), the forward's schedule.  For each key tile (chunk c, tile j) the
// item visits:
//   S  = Q K^T   (TMEM S buffer g % 2)     dP = dO V^T   (TMEM dP, released
//                                           as soon as the dS warps hold it)
//   P  = 2^(S scale log2(e) - lse log2(e))  dS = P (dP - Delta)  -> bf16 into S
//   dQ += dS K   (A = dS from TMEM, B = the K tile read MN-major)
// and dQ * scale is written as bf16 at the end of the item.
//
// CTA layout (384 threads, one CTA per SM, persistent over the schedule):
//   warps 0-7  dS in two warpgroups (thread = query row, half of the key
//              columns) and the dQ epilogue (half of the head dimension)
//   warp 8     producer: gathers the item's Q and dO rows (cp.async) and
//              issues the K tile TMA loads into a 3-slot ring
//   warp 10    producer of the V tiles (2-slot ring)
//   warp 9     TMEM allocator, S = Q K^T and dQ += dS K issuer (one thread)
//   warp 11    dP = dO V^T issuer (one thread)
// TMEM: S buffers [0,128) and [128,256), dP [256,384), dQ [384, 384+D).  A K
// slot is read by S of its tile and by dQ of that tile, so it frees after the
// dQ product; S buffer b is overwritten by an S issued after the dQ that read
// its dS, by the same thread (the tensor pipe runs one thread's MMAs in issue
// order).
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace thd {

template <int D>
struct DqCfg {
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kQBytes = kTile * D * 2;  // one [128, D] bf16 tile
  static constexpr int kKVBytes = kTile * D * 2;
  static constexpr int kSmem = 1024 + 2 * kQBytes + (kKStages + kVStages) * kKVBytes;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColDP = 256, kColDQ = 384;
  static constexpr int kThreads = 384;
  // register split (setmaxnreg) for the instantiation shorter sequences take:
  // dQ +2-3% on batches of 0.1-8K-token sequences, -0.9% on one long sequence
  static constexpr uint32_t kComputeRegs = 192;  // per thread, warps 0-7
  static constexpr uint32_t kOtherRegs = 112;    // per thread, warps 8-11
  static_assert(256 * kComputeRegs + 128 * kOtherRegs <= 384 * 168, "register split above the launch budget");
};

template <int D, bool kGrouped>
__global__ void __launch_bounds__(384, 1)
    dq_kernel(const DqParams p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = DqCfg<D>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::kQBytes;
  uint8_t* sK = smem + 2 * C::kQBytes;
  uint8_t* sV = sK + KS * C::kKVBytes;
  __shared__ __align__(8) uint64_t bar_k_full[KS];
  __shared__ __align__(8) uint64_t bar_k_empty[KS];
  __shared__ __align__(8) uint64_t bar_v_full[VS];
  __shared__ __align__(8) uint64_t bar_v_empty[VS];
  __shared__ __align__(8) uint64_t bar_s_full[2];
  __shared__ __align__(8) uint64_t bar_ds_ready[2];
  __shared__ __align__(8) uint64_t bar_dp_full;
  __shared__ __align__(8) uint64_t bar_dp_free;  // the dS warps have read dP into registers
  __shared__ __align__(8) uint64_t bar_q_full;
  __shared__ __align__(8) uint64_t bar_q_empty;
  __shared__ __align__(8) uint64_t bar_dq_done;
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ __align__(8) uint64_t bar_drain2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ ItemRing ring;  // items handed out to this CTA, in claim order

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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_ds_ready[s], 8);  // one arrival per dS warp
    }
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_dp_free, 8);  // one arrival per dS warp
    mbar_init(&bar_q_full, 32);
    mbar_init(&bar_q_empty, 2);  // the S issuer's last read of Q and the dP issuer's last read of dO
    mbar_init(&bar_dq_done, 1);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_drain2, 1);
    item_ring_init(&ring, 3 + 8);  // warps 9, 10, 11 (one thread each) and the 8 dS warps
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
  } else if (warp >= 8) {
    if constexpr (!kGrouped) regs_lower<C::kOtherRegs>();
    if (warp == 8) {
      // ------------------------------------------------------------ Q, dO and K producer (whole warp)
      int ks = 0;
      uint32_t kph = 0, n_fill = 0, q_iter = 0;
      bool ok = true;
      int w = item_first();
      for (uint32_t kit = 0; ok; ++kit) {
        // publish this item (or the end marker) to the other roles, and claim
        // the next one while this one is loaded
        int wnext = 0;
        if (lane == 0) {
          ok = item_publish(&ring, kit, w, &s_abort);
          if (ok && w < n_items) wnext = item_claim(p.claim);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok || w >= n_items) break;
        const QItem it = q_item<kGrouped>(p, n_entries, w);
        // the item's rank-local query rows of Q and dO, once the previous
        // item's last products that read them have completed; rows without a
        // valid query are zero
        if (!mbar_wait(&bar_q_empty, (q_iter & 1u) ^ 1u, &s_abort)) break;
        const uint32_t qdst = smem_u32(sQ), ddst = smem_u32(sDO);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int row = lane + 32 * rr;
          const int prow = it.t * kTile + row;
          const bool in_rank = prow < 2 * it.g.cbq;
          const int pos = in_rank ? local_to_pos(prow, it.r, it.g.cbq, p.cp) : 0;
          const bool valid = in_rank && pos < it.g.Lq;
          const int64_t off = valid ? (((int64_t)it.g.q_off + pos) * p.Hq + it.h) * D : 0;
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            cp_async_16(qdst + sw128_offset(row, 8 * c, kTile), p.q + off + (valid ? 8 * c : 0), valid ? 16u : 0u);
            cp_async_16(ddst + sw128_offset(row, 8 * c, kTile), p.dout + off + (valid ? 8 * c : 0), valid ? 16u : 0u);
          }
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&bar_q_full);
        ++q_iter;
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
        w = __shfl_sync(0xffffffffu, wnext, 0);
      }
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
          int w;
          if (!item_take_one(&ring, kit, w, &s_abort) || w >= n_items) break;
          const QItem it = q_item<kGrouped>(p, n_entries, w);
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
      // ------------------------------------------------------------ S = Q K^T and dQ += dS K issuer
      // Two issuing threads, as in the forward: a barrier wait in one does not
      // leave the tensor pipe idle while the other has products to issue.
      // This one issues, per tile g of an item, S(g) and then dQ(g-1) once the
      // dS warps have written dS(g-1) (ds_ready): S(g+1) thus follows dQ(g-1)
      // at once and is ready one tile ahead.  S(g) goes into S buffer g % 2,
      // whose dS(g-2) the dQ(g-2) issued before it by this same thread reads:
      // the tensor pipe runs one thread's MMAs in issue order, so no wait.
      if (lane == 0) {
        constexpr uint32_t idesc_dq = idesc_bf16(128, D, false, true);
        const uint64_t qdesc = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t kdesc = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t kmn = sdesc_sw128(smem_u32(sK), 16384, 1024);  // K read MN-major
        int ks = 0;
        uint32_t kph = 0, g = 0, q_iter = 0;
        bool ok = true;
        // issue dQ += dS K for tile gg (its dS in S buffer gg % 2, its K in ring slot gg % KS)
        auto issue_dq = [&](uint32_t gg, int ncols, bool first) -> bool {
          const uint32_t b = gg & 1u;
          if (!mbar_wait(&bar_ds_ready[b], (gg >> 1) & 1u, &s_abort)) return false;
          tc_fence_after();
          const int kslot = (int)(gg % KS);
          const uint64_t kd = kmn + (uint64_t)((kslot * C::kKVBytes) >> 4);
          // packed dS of key columns 16 kk.. sits at column 64 (kk/4) + 8 (kk%4)
          for (int kk = 0; kk < ncols / 16; ++kk)
            mma_ts(tmem + C::kColDQ, tmem + b * 128u + 64 * (kk >> 2) + 8 * (kk & 3),
                   kd + (uint64_t)(kk * (2048 >> 4)), idesc_dq, (first && kk == 0) ? 0u : 1u);
          tc_commit(&bar_k_empty[kslot]);  // the K slot's last reader
          return true;
        };
        for (uint32_t kit = 0; ok; ++kit) {
          int w;
          if (!item_take_one(&ring, kit, w, &s_abort) || w >= n_items) break;
          const QItem it = q_item<kGrouped>(p, n_entries, w);
          int n = 0;
          for_each_kv_tile(it, p, [&](int, int) { ++n; });
          if (!mbar_wait(&bar_q_full, q_iter & 1u, &s_abort)) break;
          ++q_iter;
          tc_fence_after();
          if (n == 0) {
            tc_commit(&bar_q_empty);
            continue;
          }
          int j = 0, prev_cols = 0;
          for_each_kv_tile(it, p, [&](int c, int jt) {
            if (!ok) return;
            const int ncols = q_tile_ncols(it, p, c, jt);
            const uint32_t b = g & 1u;
            if (!mbar_wait(&bar_k_full[ks], kph, &s_abort)) {
              ok = false;
              return;
            }
            tc_fence_after();
            const uint32_t idesc_s = idesc_bf16(128, ncols, false, false);
            const uint64_t kd = kdesc + (uint64_t)((ks * C::kKVBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
              mma_ss(tmem + b * 128u, qdesc + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(&bar_s_full[b]);
            if (j == n - 1) tc_commit(&bar_q_empty);  // the item's last read of Q
            if (++ks == KS) {
              ks = 0;
              kph ^= 1u;
            }
            if (j > 0 && !issue_dq(g - 1, prev_cols, j == 1)) {
              ok = false;
              return;
            }
            prev_cols = ncols;
            ++g;
            ++j;
          });
          if (!ok) break;
          if (!issue_dq(g - 1, prev_cols, n == 1)) break;
          tc_commit(&bar_dq_done);
        }
        tc_commit(&bar_drain);
        drain_wait(&bar_drain, 0);
      }
      __syncwarp();
    } else if (warp == 11) {
      // ------------------------------------------------------------ dP = dO V^T issuer
      // Per tile g: once the dS warps have read dP of tile g-1 into registers
      // (dp_free: early in their work on g-1), dP of tile g -- so it is ready
      // when they come to g.
      if (lane == 0) {
        const uint64_t dodesc = sdesc_sw128(smem_u32(sDO), 16, 1024);
        const uint64_t vdesc = sdesc_sw128(smem_u32(sV), 16, 1024);
        int vs = 0;
        uint32_t vph = 0, g = 0, q_iter = 0;
        bool ok = true;
        for (uint32_t kit = 0; ok; ++kit) {
          int w;
          if (!item_take_one(&ring, kit, w, &s_abort) || w >= n_items) break;
          const QItem it = q_item<kGrouped>(p, n_entries, w);
          int n = 0;
          for_each_kv_tile(it, p, [&](int, int) { ++n; });
          if (!mbar_wait(&bar_q_full, q_iter & 1u, &s_abort)) break;
          ++q_iter;
          tc_fence_after();
          if (n == 0) {
            tc_commit(&bar_q_empty);
            continue;
          }
          int j = 0;
          for_each_kv_tile(it, p, [&](int c, int jt) {
            if (!ok) return;
            const int ncols = q_tile_ncols(it, p, c, jt);
            // the dP buffer is free once the dS warps have read tile g-1's dP
            if ((g > 0 && !mbar_wait(&bar_dp_free, (g - 1) & 1u, &s_abort)) ||
                !mbar_wait(&bar_v_full[vs], vph, &s_abort)) {
              ok = false;
              return;
            }
            tc_fence_after();
            const uint32_t idesc_p = idesc_bf16(128, ncols, false, false);
            const uint64_t vd = vdesc + (uint64_t)((vs * C::kKVBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
              mma_ss(tmem + C::kColDP, dodesc + off, vd + off, idesc_p, kk > 0 ? 1u : 0u);
            }
            tc_commit(&bar_dp_full);
            tc_commit(&bar_v_empty[vs]);
            if (j == n - 1) tc_commit(&bar_q_empty);  // the item's last read of dO
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
    }
  } else {
    if constexpr (!kGrouped) regs_raise<C::kComputeRegs>();
    // ------------------------------------------------------------ dS + epilogue
    // Thread (half, row) owns query row `row` (its TMEM lane) and key columns
    // [64 half, 64 half + 64) of every tile, plus head-dim columns
    // [D/2 half, D/2 half + D/2) of dQ.
    const int half = warp >> 2;
    const int row = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    constexpr int DH = D / 2;
    const float sl2 = p.scale_log2;
    // dQ rows start at multiples of 128 bytes: 32-byte stores when dQ is 32-byte aligned
    const bool dq_v8 = (reinterpret_cast<uintptr_t>(p.dq) & 31u) == 0;
    uint32_t g = 0, n_item = 0;
    bool ok = true;
    for (uint32_t kit = 0; ok; ++kit) {
      int w;
      if (!item_take_warp(&ring, kit, w, &s_abort)) {
        ok = false;
        break;
      }
      if (w >= n_items) break;
      const QItem it = q_item<kGrouped>(p, n_entries, w);
      const int prow = it.t * kTile + row;
      const bool in_rank = prow < 2 * it.g.cbq;
      const int pos = in_rank ? local_to_pos(prow, it.r, it.g.cbq, p.cp) : 0;
      const bool valid = in_rank && pos < it.g.Lq;
      const int64_t grow = (int64_t)it.g.q_off + pos;
      // this row's lse (log2 units) and Delta; rows without a valid query mask
      // every key, so their values never matter
      const float dlt = valid ? p.delta[(int64_t)it.h * p.T_q + grow] : 0.f;
      const float lse2 = valid ? p.lse2[(int64_t)it.h * p.T_q + grow] : 0.f;
      int jl = 0;
      for_each_kv_tile(it, p, [&](int c, int j) {
        if (!ok) return;
        const uint32_t b = g & 1u;
        if (!mbar_wait(&bar_s_full[b], (g >> 1) & 1u, &s_abort) || !mbar_wait(&bar_dp_full, g & 1u, &s_abort)) {
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
        const int nch = ceil_div(q_tile_ncols(it, p, c, j), 32);
        const uint32_t scol = tmem + lane_base + b * 128u;
        const uint32_t pcol = tmem + lane_base + C::kColDP;
        // dP of this thread's two chunks first, so the buffer can take the
        // next tile's dP while dS is computed
        uint32_t dr[2][32];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          if (2 * half + kk < nch) tmem_ld32(pcol + 32 * (2 * half + kk), dr[kk]);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          if (2 * half + kk < nch) tmem_ld_wait(dr[kk]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_dp_free);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int ch = 2 * half + kk;  // this thread's 32-column chunk
          if (ch < nch) {
            uint32_t sr[32];
            tmem_ld32(scol + 32 * ch, sr);
            tmem_ld_wait(sr);
            // keys this row may not see get S = -inf: P = 0 and dS = 0
            if (__any_sync(0xffffffffu, cnt < 32 * ch + 32)) {
#pragma unroll
              for (int n = 0; n < 32; ++n)
                if (32 * ch + n >= cnt) sr[n] = __float_as_uint(-INFINITY);
            }
            uint32_t pk[16];
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              float x0, x1, t0, t1, g0, g1;
              ffma2(x0, x1, __uint_as_float(sr[2 * n]), __uint_as_float(sr[2 * n + 1]), sl2, sl2, -lse2, -lse2);
              const float p0 = ex2(x0), p1 = ex2(x1);
              fadd2(t0, t1, __uint_as_float(dr[kk][2 * n]), __uint_as_float(dr[kk][2 * n + 1]), -dlt, -dlt);
              fmul2(g0, g1, p0, p1, t0, t1);
              pk[n] = pack_bf16x2(g0, g1);
            }
            // packed dS stays inside this half's own S columns (the other
            // warpgroup may still be reading its half): chunk ch -> 64 (ch/2) + 16 (ch%2)
            tmem_st16(scol + 64 * (ch >> 1) + 16 * (ch & 1), pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();  // every lane's dS is in TMEM and dP was read: one arrival speaks for the warp
        if (lane == 0) mbar_arrive(&bar_ds_ready[b]);  // dS of tile g is in TMEM
        ++g;
        ++jl;
      });
      if (!ok) break;
      // ---- epilogue: dQ * scale as bf16; zero on rows without a valid query
      if (jl > 0) {
        if (!mbar_wait(&bar_dq_done, n_item & 1u, &s_abort)) break;
        tc_fence_after();
        ++n_item;
      }
#pragma unroll 1
      for (int k = 0; k < DH / 32; ++k) {
        uint32_t o[32];
        if (jl > 0) {
          tmem_ld32(tmem + lane_base + C::kColDQ + half * DH + 32 * k, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int n = 0; n < 32; ++n) o[n] = 0u;
        }
        if (in_rank)
          store32_bf16(p.dq + (grow * p.Hq + it.h) * D + half * DH + 32 * k, o, valid ? p.scale : 0.f, dq_v8);
      }
      tc_fence_before();
    }
    // ---- dQ rows past the last sequence (the slack up to dq_rows): zero
    if (ok) {
      const int Tend = p.eff[(p.B + 1) + p.B];
      const int64_t nvec = (p.dq_rows - Tend) * (int64_t)p.Hq * (D / 8);
      const int64_t base = (int64_t)Tend * p.Hq * D;
      for (int64_t i = (int64_t)blockIdx.x * 256 + tid; i < nvec; i += (int64_t)gridDim.x * 256)
        reinterpret_cast<uint4*>(p.dq + base)[i] = make_uint4(0, 0, 0, 0);
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

template <int D, bool kGrouped>
static cudaError_t launch_dq_t(const DqParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                               cudaStream_t st) {
  using C = DqCfg<D>;
  cudaError_t ea = cudaFuncSetAttribute(dq_kernel<D, kGrouped>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (ea != cudaSuccess) return ea;
  prof_before(THD_KERNEL_BWD_DQ, st);
  dq_kernel<D, kGrouped><<<grid, C::kThreads, C::kSmem, st>>>(p, tk, tv);
  count_launch();
  cudaError_t e = cudaGetLastError();
  prof_after(THD_KERNEL_BWD_DQ, st);
  return e;
}

cudaError_t launch_dq(const DqParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int D, bool grouped, int grid,
                      cudaStream_t st) {
  if (D == 128) return grouped ? launch_dq_t<128, true>(p, tk, tv, grid, st) : launch_dq_t<128, false>(p, tk, tv, grid, st);
  return grouped ? launch_dq_t<64, true>(p, tk, tv, grid, st) : launch_dq_t<64, false>(p, tk, tv, grid, st);
}

}  // namespace thd
