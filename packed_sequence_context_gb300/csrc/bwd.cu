// dK and dV of attention over packed THD tensors, key/value-stationary,
// walked in P2P ring order and executed for every emulated rank on one GB300.
//
// [P2] TransformerEngine issue #3487 ("Steps/Code to reproduce bug": BF16
// attention forward/backward on this layout with four-rank P2P context
// parallelism; "Describe the bug": THD dQ/dK/dV tail-zeroing).  [P1]
// TransformerEngine issue #2208 (traceback through AttnFuncWithCPAndKVP2P):
// in the ring, the KV of owner rank s is seen by rank r = (s + i) mod cp at
// step i, and dK/dV travel back around the ring to their owner.  Here the
// owner keeps its key tile in shared memory and visits, in ring order, the
// query tiles of every rank that sees it; dK/dV accumulate in TMEM (no
// travel).  dQ is the query-stationary pass of dq.cu.
//
// One work item = (sequence b, key chunk c, key tile jk within the chunk, kv
// head hk).  For each query tile (chunk qc, tile jq) that sees it and each
// query head h of the GQA group:
//   S^T  = K Q^T      dP^T = V dO^T     (two TMEM buffers, roles swapped every step)
//   P^T  = exp(S^T scale - lse)          dS^T = P^T (dP^T - Delta)
//   dV  += P^T dO     dK  += dS^T Q       (A = P^T / dS^T from TMEM, packed bf16
//                                          over the S^T they were computed from)
// CTA: warps 0-7 compute in two warpgroups -- a thread owns one key row (its
// TMEM lane) and half of the query columns for P/dS, and half of the head
// dimension when writing dK/dV; warp 8 TMA producer (+ lse/Delta staging);
// warp 9 TMEM allocator and S^T issuer; warp 10 dV/dK/dP^T issuer.  The
// entry-major instantiation (shorter sequences) runs 384 threads: warp 11,
// idle, completes the fourth warpgroup so that setmaxnreg can move registers
// to the compute warps (dK/dV +5% on batches of 0.1-8K-token sequences); the
// grouped one (long sequences, where that measured -1%) runs 352.
#include "common.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace thd {

template <int D>
struct BwdCfg {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = kTile * D * 2;  // one [128, D] bf16 tile
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;                 // stage s: Q at kOffQ + s * 2 * kTileBytes
  static constexpr int kOffLse = kOffQ + kStages * 2 * kTileBytes;  // stage s: lse2[128], delta[128]
  static constexpr int kOffBar = kOffLse + kStages * 2 * kTile * 4;
  static constexpr int kOffRing = kOffBar + 256;  // the item hand-out ring
  static constexpr int kSmem = kOffRing + 256;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColDV = 0, kColDK = D, kColX = 2 * D, kColY = 2 * D + 128;
  static constexpr uint32_t kComputeRegs = 200;  // per thread, warps 0-7
  static constexpr uint32_t kOtherRegs = 96;     // per thread, warps 8-11
  static_assert(256 * kComputeRegs + 128 * kOtherRegs <= 384 * 168, "register split above the launch budget");
};

struct BwdItem {
  SeqGeom g;
  int b, c, jk, hk;
  int kv_first, kv_last;  // valid key positions of the tile (first > last: none)
};

// Work item w -> (schedule entry, kv head).  Items are ordered by groups of
// p.group_kv kv heads (outermost: while a group runs, the queries and output
// gradients of its query heads are what the CTAs read, so they stay in L2),
// then by schedule entry (longest first), then by the group's kv heads.
template <bool kGrouped>
__device__ inline BwdItem bwd_item(const BwdParams& p, int n_entries, int w) {
  BwdItem it;
  int4 e;
  if constexpr (kGrouped) {
    const int per = n_entries * p.group_kv;  // items per group
    const int grp = w / per, rem = w - grp * per;
    e = p.items[rem / p.group_kv];
    it.hk = grp * p.group_kv + rem % p.group_kv;
  } else {  // one group: entry-major, kv heads innermost
    (void)n_entries;
    e = p.items[w / p.Hkv];
    it.hk = w % p.Hkv;
  }
  it.b = e.x;
  it.c = e.y;
  it.jk = e.z;
  it.g = seq_geom(p.eff, p.B, it.b, p.cp, p.causal);
  bwd_kv_range(it.g, it.c, it.jk, it.kv_first, it.kv_last);
  return it;
}

// Calls f(qc, jq, h) for every (query tile, query head) that sees the item's
// key tile, in ring order of the ranks holding the key tile.
template <typename F>
__device__ inline void for_each_q_step(const BwdItem& it, const BwdParams& p, F&& f) {
  if (it.kv_first > it.kv_last) return;
  const int G = p.Hq / p.Hkv;
  const int s = chunk_owner(it.c, p.cp);
  const int nq = ceil_div(it.g.cbq, kTile);
  for (int i = 0; i < p.cp; ++i) {
    const int r = (s + i) % p.cp;
    for (int e = 0; e < 2; ++e) {
      const int qc = e == 0 ? r : 2 * p.cp - 1 - r;
      for (int jq = 0; jq < nq; ++jq) {
        if (!bwd_q_tile_visits(it.g, qc, jq, it.kv_first, it.kv_last, p.causal != 0)) continue;
        for (int hh = 0; hh < G; ++hh) f(qc, jq, it.hk * G + hh);
      }
    }
  }
}

__device__ inline void drain_wait_b(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitTimeoutNs) break;
  }
}

template <int D, bool kGrouped>
__global__ void __launch_bounds__(kGrouped ? 352 : 384, 1)
    bwd_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = BwdCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);  // stage s: [s*256, s*256+128) lse2, then delta
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* bar_kv_full = bars + 0;
  uint64_t* bar_kv_empty = bars + 1;
  uint64_t* bar_qdo_full = bars + 2;       // [S] Q (TMA) and lse / Delta (cp.async) of the stage landed
  uint64_t* bar_qdo_empty = bars + 2 + S;  // [S] the stage's Q may be refilled (its dK completed)
  uint64_t* bar_st_full = bars + 2 + 2 * S;
  uint64_t* bar_p_ready = bars + 3 + 2 * S;
  uint64_t* bar_dk_done = bars + 4 + 2 * S;
  uint64_t* bar_y_free = bars + 5 + 2 * S;  // the compute warps hold dP^T in registers
  uint64_t* bar_dp_full = bars + 10 + 2 * S;  // dP^T of the step is in TMEM
  uint64_t* bar_drain = bars + 6 + 2 * S;
  uint64_t* bar_drain2 = bars + 11 + 2 * S;
  uint64_t* bar_do_full = bars + 12 + 2 * S;   // [S] dO of the stage landed (TMA)
  uint64_t* bar_do_empty = bars + 12 + 3 * S;  // [S] the stage's dO may be refilled (its dV completed)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 8 + 2 * S);
  int* s_abort = reinterpret_cast<int*>(bars + 9 + 2 * S);
  ItemRing* ring = reinterpret_cast<ItemRing*>(smem + C::kOffRing);  // items of this CTA, in claim order

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (*p.dev_status != 0) return;
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
    if (tid == 0) atomicCAS(p.dev_status, 0, THD_ERR_UNSUPPORTED);
    return;
  }
  const int n_entries = p.counters[0];
  const int n_items = n_entries * p.Hkv;

  if (tid == 0) {
    mbar_init(bar_kv_full, 1);
    mbar_init(bar_kv_empty, 2);  // warp 9 saw the tile arrive; warp 10: its last reader completed
    for (int s = 0; s < S; ++s) {
      mbar_init(&bar_qdo_full[s], 33);  // 32 cp.async arrivals + the TMA expect-tx arrival
      mbar_init(&bar_qdo_empty[s], 1);
      mbar_init(&bar_do_full[s], 1);
      mbar_init(&bar_do_empty[s], 1);
    }
    mbar_init(bar_st_full, 1);
    mbar_init(bar_p_ready, 8);  // one arrival per compute warp
    mbar_init(bar_dk_done, 1);
    mbar_init(bar_y_free, 8);  // one arrival per compute warp
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_drain2, 1);
    mbar_init(bar_drain, 1);
    item_ring_init(ring, 2 + 8);  // warps 9, 10 (one thread each) and the 8 compute warps
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // Test hook (thd_test_arm_stall): every thread waits on a barrier nothing
  // completes, so the bounded wait runs out, the CTA takes the abort path
  // before any copy or MMA is issued, frees its TMEM and reports
  // THD_ERR_TIMEOUT.  The drain barrier is free for this: in this mode no
  // role runs, so nothing ever commits to it.
  if (p.test_stall) {
    mbar_wait(bar_drain, 0, s_abort);
  } else if (warp >= 8) {
    // The compute warps hold a step's P (64 values) and S^T / dP^T chunks per
    // thread: they get 200 registers, warps 8-11 (producer, issuers, idle) 96;
    // 256 x 200 + 128 x 96 fits the 384 x 168 the CTA is launched with.
    if constexpr (!kGrouped) regs_lower<C::kOtherRegs>();
    if (warp == 8) {
      // ------------------------------------------------------------ producer (whole warp)
      int stage = 0;
      uint32_t ph = 0, kv_iter = 0, n_fill = 0;
      bool ok = true;
      int w = item_first();
      for (uint32_t kit = 0; ok; ++kit, w = __shfl_sync(0xffffffffu, w, 0)) {
        // publish this item (or the end marker) to the other roles, and claim
        // the next one (lane 0's w) while this one is loaded
        int wcur = w;
        if (lane == 0) {
          ok = item_publish(ring, kit, wcur, s_abort);
          if (ok && wcur < n_items) w = item_claim(p.claim);
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok || wcur >= n_items) break;
        const BwdItem it = bwd_item<kGrouped>(p, n_entries, wcur);
        if (it.kv_first > it.kv_last) continue;  // no valid key: nothing to load
        const int kv_row = it.g.kv_off + it.c * it.g.cbkv + it.jk * kTile;
        if (!mbar_wait(bar_kv_empty, (kv_iter & 1u) ^ 1u, s_abort)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_kv_full, 2 * C::kTileBytes);
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb) {
            tma_load_3d(smem_u32(sK + hb * 16384), &tmK, bar_kv_full, hb * 64, it.hk, kv_row);
            tma_load_3d(smem_u32(sV + hb * 16384), &tmV, bar_kv_full, hb * 64, it.hk, kv_row);
          }
        }
        ++kv_iter;
        for_each_q_step(it, p, [&](int qc, int jq, int h) {
          if (!ok) return;
          if (!mbar_wait(&bar_qdo_empty[stage], ph ^ 1u, s_abort)) {
            ok = false;
            return;
          }
          const int q0 = qc * it.g.cbq + jq * kTile;
          const int nqv = imin(imin(kTile, it.g.cbq - jq * kTile), it.g.Lq - q0);
          const int q_row = it.g.q_off + q0;
          const uint32_t lse_st = smem_u32(sLse + stage * 256);
          // lse and Delta of the valid query rows, copied asynchronously; the
          // entries past nqv are zeroed so that masked columns stay finite
          // (S = -inf gives P = 0 and dS = 0 only against finite lse and Delta)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = lane + 32 * k;
            if (n < nqv) {
              const int64_t idx = (int64_t)h * p.T_q + q_row + n;
              cp_async_4(lse_st + 4 * n, p.lse2 + idx);
              cp_async_4(lse_st + 512 + 4 * n, p.delta + idx);
            } else {
              sLse[stage * 256 + n] = 0.f;
              sLse[stage * 256 + 128 + n] = 0.f;
            }
          }
          cp_async_arrive_noinc(&bar_qdo_full[stage]);
          __syncwarp();  // the zeroed entries are ordered before lane 0's arrival
          uint8_t* sQ = smem + C::kOffQ + stage * 2 * C::kTileBytes;
          uint8_t* sDO = sQ + C::kTileBytes;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bar_qdo_full[stage], C::kTileBytes);
#pragma unroll
            for (int hb = 0; hb < D / 64; ++hb)
              tma_load_3d(smem_u32(sQ + hb * 16384), &tmQ, &bar_qdo_full[stage], hb * 64, h, q_row);
          }
          // dO has its own release: its last reader (dV) completes after Q's (dK)
          if (!mbar_wait(&bar_do_empty[stage], ph ^ 1u, s_abort)) {
            ok = false;
            return;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&bar_do_full[stage], C::kTileBytes);
#pragma unroll
            for (int hb = 0; hb < D / 64; ++hb)
              tma_load_3d(smem_u32(sDO + hb * 16384), &tmDO, &bar_do_full[stage], hb * 64, h, q_row);
          }
          ++n_fill;
          if (++stage == S) {
            stage = 0;
            ph ^= 1u;
          }
        });
      }
      // every issued copy must land before the CTA may exit
      if (kv_iter > 0) drain_wait_b(bar_kv_full, (kv_iter - 1) & 1u);
      for (int s = 0; s < S; ++s) {
        const uint32_t fills = n_fill > (uint32_t)s ? (n_fill - 1 - s) / S + 1 : 0;
        if (fills > 0) {
          drain_wait_b(&bar_qdo_full[s], (fills - 1) & 1u);
          drain_wait_b(&bar_do_full[s], (fills - 1) & 1u);
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------ S^T issuer
      // The two 128-column TMEM buffers T0, T1 swap roles every step: step s
      // puts S^T(s) (then P^T(s)) in T[s % 2] and dP^T(s) in T[(s + 1) % 2].
      // Two issuing threads, as in the forward (a barrier wait in one does not
      // idle the tensor pipe while the other has products to issue):
      //   warp 9:  S^T(s), as soon as the compute warps hold dP^T(s-1), which sat
      //            in the same buffer, in registers (y_free)
      //   warp 10: once the compute warps have written P^T(s-1) and dS(s-1),
      //            dV(s-1) and dK(s-1); then dP^T(s) into the buffer P^T(s-1)
      //            leaves once dV(s-1) has read it.
      // The compute warps of step s compute P from S^T(s) while dV/dK(s-1) run
      // and dS once dP^T(s) is there.  P^T(s) and dS^T(s) both go back over
      // S^T(s) as packed bf16 (each thread into the S^T columns it has read) and
      // are the TMEM A operands of dV(s) and dK(s): dS never touches shared
      // memory, which the SS products already keep busy.
      if (lane == 0) {
        const uint32_t kb = smem_u32(sK);
        int stage = 0;
        uint32_t ph = 0, su = 0, kv_iter = 0;
        bool ok = true;
        for (uint32_t kit = 0; ok; ++kit) {
          int w;
          if (!item_take_one(ring, kit, w, s_abort) || w >= n_items) break;
          const BwdItem it = bwd_item<kGrouped>(p, n_entries, w);
          if (it.kv_first > it.kv_last) continue;
          if (!mbar_wait(bar_kv_full, kv_iter & 1u, s_abort)) break;
          ++kv_iter;
          // this thread has seen the tile's phase: the tile may be refilled once
          // warp 10 also releases it, and never before this wait (which would
          // leave this wait two phases behind when the item has no step)
          mbar_arrive(bar_kv_empty);
          for_each_q_step(it, p, [&](int qc, int jq, int) {
            if (!ok) return;
            const int nqv = imin(imin(kTile, it.g.cbq - jq * kTile), it.g.Lq - (qc * it.g.cbq + jq * kTile));
            const uint32_t idesc_t = idesc_bf16(128, 16 * ceil_div(nqv, 16), false, false);
            const uint32_t acol = tmem + C::kColX + 128u * (su & 1u);  // S^T(s), then P^T(s)
            if (!mbar_wait(&bar_qdo_full[stage], ph, s_abort) ||
                (su > 0 && !mbar_wait(bar_y_free, (su - 1) & 1u, s_abort))) {
              ok = false;
              return;
            }
            tc_fence_after();
            const uint32_t qb = smem_u32(smem + C::kOffQ + stage * 2 * C::kTileBytes);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
              mma_ss(acol, sdesc_sw128(kb + off, 16, 1024), sdesc_sw128(qb + off, 16, 1024), idesc_t, ks > 0);
            }
            tc_commit(bar_st_full);
            ++su;
            if (++stage == S) {
              stage = 0;
              ph ^= 1u;
            }
          });
        }
        tc_commit(bar_drain);
        drain_wait_b(bar_drain, 0);
      }
      __syncwarp();
    } else if (warp == 10) {
      // ------------------------------------------------------------ dV, dK and dP^T issuer
      if (lane == 0) {
        constexpr uint32_t idesc_kv = idesc_bf16(128, D, false, true);  // dV, dK (B MN-major)
        const uint32_t vb = smem_u32(sV);
        int stage = 0;
        uint32_t ph = 0, su = 0, kv_iter = 0;
        bool ok = true;
        // the step whose dV / dK are still to be issued
        int pv_stage = -1, pv_n16 = 0;
        bool pv_first = false;
        auto tail = [&](bool last) -> bool {
          const uint32_t ps = su - 1;  // the pending step
          if (!mbar_wait(bar_p_ready, ps & 1u, s_abort)) return false;
          // The compute warps wrote P^T and dS^T of the item's last step only
          // after its S^T and dP^T -- the last products that read K and V --
          // had completed: the K/V tile may be refilled with the next item's
          // while the last dV and dK run and the epilogue drains them.
          if (last) mbar_arrive(bar_kv_empty);
          tc_fence_after();
          const uint32_t qb = smem_u32(smem + C::kOffQ + pv_stage * 2 * C::kTileBytes);
          const uint32_t dob = qb + C::kTileBytes;
          const uint32_t pcol = tmem + C::kColX + 128u * (ps & 1u);  // P^T of the pending step
          // dK first: its completion frees the stage's Q, which the S^T two
          // steps on waits for, one product earlier than dO.
          // dK += dS^T Q  (dS^T packed bf16 beside P^T: K-step ks at column
          // 64 (ks/4) + 32 + 8 (ks%4); K = the valid query rows)
          for (int ks = 0; ks < pv_n16; ++ks)
            mma_ts(tmem + C::kColDK, pcol + 64 * (ks >> 2) + 32 + 8 * (ks & 3), sdesc_sw128(qb + ks * 2048, 16384, 1024),
                   idesc_kv, (pv_first && ks == 0) ? 0u : 1u);
          tc_commit(&bar_qdo_empty[pv_stage]);
          // dV += P^T dO  (P^T packed bf16: query columns 16 ks.. of K-step ks sit
          // at column 64 (ks/4) + 8 (ks%4))
          for (int ks = 0; ks < pv_n16; ++ks)
            mma_ts(tmem + C::kColDV, pcol + 64 * (ks >> 2) + 8 * (ks & 3), sdesc_sw128(dob + ks * 2048, 16384, 1024),
                   idesc_kv, (pv_first && ks == 0) ? 0u : 1u);
          tc_commit(&bar_do_empty[pv_stage]);
          // the item's last step: dk_done completes once per item, when every
          // product of the item has (this thread's MMAs complete in order)
          if (last) tc_commit(bar_dk_done);
          pv_stage = -1;
          return true;
        };
        for (uint32_t kit = 0; ok; ++kit) {
          int w;
          if (!item_take_one(ring, kit, w, s_abort) || w >= n_items) break;
          const BwdItem it = bwd_item<kGrouped>(p, n_entries, w);
          if (it.kv_first > it.kv_last) continue;
          if (!mbar_wait(bar_kv_full, kv_iter & 1u, s_abort)) break;
          ++kv_iter;
          tc_fence_after();
          bool first = true;
          for_each_q_step(it, p, [&](int qc, int jq, int) {
            if (!ok) return;
            const int nqv = imin(imin(kTile, it.g.cbq - jq * kTile), it.g.Lq - (qc * it.g.cbq + jq * kTile));
            const int n16 = ceil_div(nqv, 16);
            const uint32_t idesc_t = idesc_bf16(128, 16 * n16, false, false);
            const uint32_t bcol = tmem + C::kColX + 128u * ((su + 1) & 1u);  // dP^T(s)
            if (!mbar_wait(&bar_qdo_full[stage], ph, s_abort)) {
              ok = false;
              return;
            }
            // dV, dK of the previous step (of this item; an item's last step is
            // finished at the item's end)
            if (pv_stage >= 0 && !tail(false)) {
              ok = false;
              return;
            }
            // dP^T = V dO^T -> the buffer P^T(s-1) and dS^T(s-1) leave once dV(s-1)
            // and dK(s-1) have read them: this thread issued those just before,
            // and the tensor pipe executes one thread's MMAs in issue order
            if (!mbar_wait(&bar_do_full[stage], ph, s_abort)) {
              ok = false;
              return;
            }
            tc_fence_after();
            const uint32_t dob = smem_u32(smem + C::kOffQ + stage * 2 * C::kTileBytes) + C::kTileBytes;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
              mma_ss(bcol, sdesc_sw128(vb + off, 16, 1024), sdesc_sw128(dob + off, 16, 1024), idesc_t, ks > 0);
            }
            tc_commit(bar_dp_full);
            pv_stage = stage;
            pv_n16 = n16;
            pv_first = first;
            first = false;
            ++su;
            if (++stage == S) {
              stage = 0;
              ph ^= 1u;
            }
          });
          if (!ok) break;
          if (pv_stage >= 0) {
            if (!tail(true)) break;  // the item's last step; dk_done then covers all its products
          } else {
            mbar_arrive(bar_kv_empty);  // no step read the tile
          }
        }
        tc_commit(bar_drain2);
        drain_wait_b(bar_drain2, 0);
      }
      __syncwarp();
    }
  } else {
    if constexpr (!kGrouped) regs_raise<C::kComputeRegs>();
    // ------------------------------------------------------------ compute warps
    const int half = warp >> 2;     // which half of the columns this thread owns
    const int row = tid & 127;      // its key row (TMEM lane) / query row when draining dQ
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    // dK/dV rows start at multiples of 128 bytes: with 32-byte aligned buffers
    // the epilogue stores whole 32-byte sectors (the API asks for 16)
    const bool v8_ok = ((reinterpret_cast<uintptr_t>(p.dk) | reinterpret_cast<uintptr_t>(p.dv)) & 31u) == 0;
    uint32_t su = 0, n_done = 0;
    bool ok = true;
    for (uint32_t kit = 0; ok; ++kit) {
      int w;
      if (!item_take_warp(ring, kit, w, s_abort)) {
        ok = false;
        break;
      }
      if (w >= n_items) break;
      const BwdItem it = bwd_item<kGrouped>(p, n_entries, w);
      const int kv_local = it.jk * kTile + row;  // row within the chunk
      const int j_pos = it.c * it.g.cbkv + kv_local;
      const bool in_chunk = kv_local < it.g.cbkv;
      const bool valid_kv = in_chunk && j_pos < it.g.Lkv;
      int nsteps = 0;
      for_each_q_step(it, p, [&](int qc, int jq, int h) {
        if (!ok) return;
        if (!mbar_wait(bar_st_full, su & 1u, s_abort)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const int q0 = qc * it.g.cbq + jq * kTile;
        const int nqv = imin(imin(kTile, it.g.cbq - jq * kTile), it.g.Lq - q0);
        int n_lo = 0, n_hi = valid_kv ? nqv : 0;
        if (p.causal) n_lo = imin(imax(j_pos - it.g.koff - q0, 0), kTile);
        // the cp.async writes of lse/Delta are visible to the threads that
        // observe the stage barrier's phase, so observe it here (it cannot have
        // moved on: the stage is refilled only after this step's p_ready)
        if (!mbar_wait(&bar_qdo_full[su % S], (su / S) & 1u, s_abort)) {
          ok = false;
          return;
        }
        const uint32_t lse_s = smem_u32(sLse + (su % S) * 256), dl_s = lse_s + 512;
        const int nch = ceil_div(nqv, 32);
        const uint32_t acol = tmem + lane_base + C::kColX + 128u * (su & 1u);        // S^T, then P^T
        const uint32_t bcol = tmem + lane_base + C::kColX + 128u * ((su + 1) & 1u);  // dP^T
        // ---- P = 2^(S^T scale log2(e) - lse) for this thread's chunks (query
        // columns outside [n_lo, n_hi) -- causal, or past the valid rows -- get
        // S = -inf, hence P = 0 and dS = 0); packed P^T goes back over S^T
        float pv[2][32];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int kk = 2 * half + i;
          if (kk < nch) {
            uint32_t sr[32];
            tmem_ld32(acol + 32 * kk, sr);
            tmem_ld_wait(sr);
            if (__any_sync(0xffffffffu, n_lo > 32 * kk || n_hi < 32 * kk + 32)) {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int n = 32 * kk + e;
                if (n < n_lo || n >= n_hi) sr[e] = __float_as_uint(-INFINITY);
              }
            }
            uint32_t pk[16];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 l4 = lds128f(lse_s + 4 * (32 * kk + 4 * q4));  // lse in log2 units
              float x0, x1, x2, x3;
              ffma2(x0, x1, __uint_as_float(sr[4 * q4]), __uint_as_float(sr[4 * q4 + 1]), sl2, sl2, -l4.x, -l4.y);
              ffma2(x2, x3, __uint_as_float(sr[4 * q4 + 2]), __uint_as_float(sr[4 * q4 + 3]), sl2, sl2, -l4.z, -l4.w);
              pv[i][4 * q4] = ex2(x0);
              pv[i][4 * q4 + 1] = ex2(x1);
              pv[i][4 * q4 + 2] = ex2(x2);
              pv[i][4 * q4 + 3] = ex2(x3);
              pk[2 * q4] = pack_bf16x2(pv[i][4 * q4], pv[i][4 * q4 + 1]);
              pk[2 * q4 + 1] = pack_bf16x2(pv[i][4 * q4 + 2], pv[i][4 * q4 + 3]);
            }
            // packed P^T stays inside this warpgroup's own S^T columns (the other
            // warpgroup may still be reading its half): chunk kk -> 64 (kk/2) + 16 (kk%2)
            tmem_st16(acol + 64 * (kk >> 1) + 16 * (kk & 1), pk);
          }
        }
        // ---- dS = P (dP^T - Delta), once dP^T is in TMEM; the buffer is
        // released (y_free) as soon as this warp's last chunk of it is loaded
        if (!mbar_wait(bar_dp_full, su & 1u, s_abort)) {
          ok = false;
          return;
        }
        tc_fence_after();
        if (2 * half >= nch) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_y_free);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int kk = 2 * half + i;
          if (kk < nch) {
            uint32_t dr[32];
            tmem_ld32(bcol + 32 * kk, dr);
            tmem_ld_wait(dr);
            if (kk + 1 >= imin(nch, 2 * half + 2)) {  // this warp's last dP^T chunk is in registers
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_y_free);
            }
            uint32_t dk[16];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 d4 = lds128f(dl_s + 4 * (32 * kk + 4 * q4));
              float t0, t1, t2, t3, g0, g1, g2, g3;
              fadd2(t0, t1, __uint_as_float(dr[4 * q4]), __uint_as_float(dr[4 * q4 + 1]), -d4.x, -d4.y);
              fadd2(t2, t3, __uint_as_float(dr[4 * q4 + 2]), __uint_as_float(dr[4 * q4 + 3]), -d4.z, -d4.w);
              fmul2(g0, g1, pv[i][4 * q4], pv[i][4 * q4 + 1], t0, t1);
              fmul2(g2, g3, pv[i][4 * q4 + 2], pv[i][4 * q4 + 3], t2, t3);
              dk[2 * q4] = pack_bf16x2(g0, g1);
              dk[2 * q4 + 1] = pack_bf16x2(g2, g3);
            }
            // packed dS^T beside P^T, in the S^T columns this thread has read:
            // chunk kk -> 64 (kk/2) + 32 + 16 (kk%2)
            tmem_st16(acol + 64 * (kk >> 1) + 32 + 16 * (kk & 1), dk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();  // every lane's P^T and dS^T are in TMEM: one arrival speaks for the warp
        if (lane == 0) mbar_arrive(bar_p_ready);
        ++su;
        ++nsteps;
      });
      if (!ok) break;
      // ---- epilogue: dK (scaled) and dV of this key tile, zeros on pad rows,
      // once the item's last dK (and with it every product before) completed
      if (nsteps > 0) {
        if (!mbar_wait(bar_dk_done, n_done & 1u, s_abort)) break;  // one phase per item with steps
        ++n_done;
        tc_fence_after();
      }
#pragma unroll 1
      for (int kk = half * (D / 64); kk < (half + 1) * (D / 64); ++kk) {
        uint32_t a[32], bq[32];
        if (nsteps > 0) {
          tmem_ld32(tmem + lane_base + C::kColDK + 32 * kk, a);
          tmem_ld32(tmem + lane_base + C::kColDV + 32 * kk, bq);
          tmem_ld_wait(a);
          tmem_ld_wait(bq);
        } else {
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            a[n] = 0u;
            bq[n] = 0u;
          }
        }
        if (in_chunk) {
          const float fk = valid_kv ? p.scale : 0.f;
          const float fv = valid_kv ? 1.f : 0.f;
          const int64_t grow = (int64_t)it.g.kv_off + j_pos;
          uint16_t* dkp = p.dk + (grow * p.Hkv + it.hk) * D + 32 * kk;
          uint16_t* dvp = p.dv + (grow * p.Hkv + it.hk) * D + 32 * kk;
          uint32_t x[16], y[16];  // the 32 columns of dK and of dV, packed bf16
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            x[n] = pack_bf16x2(__uint_as_float(a[2 * n]) * fk, __uint_as_float(a[2 * n + 1]) * fk);
            y[n] = pack_bf16x2(__uint_as_float(bq[2 * n]) * fv, __uint_as_float(bq[2 * n + 1]) * fv);
          }
          if (v8_ok) {
            // two 32-byte stores per tensor: each writes one whole sector of the row
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              st_global_v8(dkp + 16 * h2, *reinterpret_cast<const uint32_t(*)[8]>(x + 8 * h2));
              st_global_v8(dvp + 16 * h2, *reinterpret_cast<const uint32_t(*)[8]>(y + 8 * h2));
            }
          } else {
#pragma unroll
            for (int n = 0; n < 4; ++n) {
              reinterpret_cast<uint4*>(dkp)[n] = make_uint4(x[4 * n], x[4 * n + 1], x[4 * n + 2], x[4 * n + 3]);
              reinterpret_cast<uint4*>(dvp)[n] = make_uint4(y[4 * n], y[4 * n + 1], y[4 * n + 2], y[4 * n + 3]);
            }
          }
        }
      }
      tc_fence_before();
    }
    // ---- dK/dV rows past the last sequence: zero
    if (ok) {
      const int Tend = p.eff[3 * (p.B + 1) + p.B];
      const int64_t nvec = (p.dkv_rows - Tend) * (int64_t)p.Hkv * (D / 8);
      const int64_t base = (int64_t)Tend * p.Hkv * D;
      for (int64_t i = (int64_t)blockIdx.x * 256 + tid; i < nvec; i += (int64_t)gridDim.x * 256) {
        reinterpret_cast<uint4*>(p.dk + base)[i] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(p.dv + base)[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && *s_abort) atomicCAS(p.dev_status, 0, THD_ERR_TIMEOUT);
}

template <int D, bool kGrouped>
static cudaError_t launch_bwd_t(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                                const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t st) {
  using C = BwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D, kGrouped>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  prof_before(THD_KERNEL_BWD, st);
  bwd_kernel<D, kGrouped><<<grid, kGrouped ? 352 : 384, C::kSmem, st>>>(p, tq, tdo, tk, tv);
  count_launch();
  e = cudaGetLastError();
  prof_after(THD_KERNEL_BWD, st);
  return e;
}

cudaError_t launch_bwd(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                       const CUtensorMap& tv, int D, bool grouped, int grid, cudaStream_t st) {
  if (D == 128)
    return grouped ? launch_bwd_t<128, true>(p, tq, tdo, tk, tv, grid, st)
                   : launch_bwd_t<128, false>(p, tq, tdo, tk, tv, grid, st);
  return grouped ? launch_bwd_t<64, true>(p, tq, tdo, tk, tv, grid, st)
                 : launch_bwd_t<64, false>(p, tq, tdo, tk, tv, grid, st);
}

}  // namespace thd
