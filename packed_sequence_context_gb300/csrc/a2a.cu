// The all-to-all of an emulated Ulysses (A2A) or hierarchical a2a+p2p
// context-parallel layer, every rank and group in one launch.
//
// Pages: TransformerEngine issue #2208, "thd format is not supported with
// hierarchical CP implementation yet" (the maintainer's reply: A2A versus
// P2P, and THD lacking A2A); "Hybrid / Hierarchical Context Parallel Skill"
// (a2a+p2p with hierarchical sizes [a2a, p2p] whose product is the CP size;
// "Contraintes requises": padded lengths divisible by 2 * cp).
//
// Layouts (no layout is printed on the pages; the plainest reading):
//   shards  [cp][T/cp, H, D]: CP rank r's THD shard, rank-local rows in the
//           load-balanced order (chunk r then chunk 2cp-1-r of every
//           sequence, chunk = P_b / (2 cp) rows);
//   groups  [a2a][T, H/a2a, D]: member i of the a2a groups holds heads
//           [i H/a2a, (i+1) H/a2a) of every token at its global padded row.
// Groups are runs of a2a consecutive ranks, so group j holds exactly the rows
// p2p rank j owns under the 2 p2p split; the P2P ring across groups then runs
// on each member's tensor in global order.
//
// The copy is a permutation of rows: one warp per global token, 16-byte
// vector loads and stores, kA2aUnroll vectors per lane in flight.
#include "a2a.cuh"

namespace thd {

constexpr int kA2aThreads = 256;
constexpr int kA2aUnroll = 4;

// Largest b in [0, B] with pad[b] <= g (pad non-decreasing, pad[0] = 0 <= g),
// then past any empty sequences that share the offset.
__device__ inline int a2a_seq_of(const int32_t* pad, int B, int g) {
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pad[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  while (lo < B && pad[lo + 1] <= g) ++lo;
  return lo;
}

template <bool kToGroups>
__global__ void __launch_bounds__(kA2aThreads) a2a_kernel(A2aParams p) {
  if (*p.dev_status != 0) return;  // metadata rejected: outputs untouched
  const int lane = threadIdx.x & 31;
  const int B = p.B, cp = p.cp;
  const int Tend = p.pad[B];  // rows past the last sequence are not moved
  const int64_t rows_rank = p.T / cp;
  const int wpb = kA2aThreads / 32;
  for (int g = blockIdx.x * wpb + (threadIdx.x >> 5); g < Tend; g += gridDim.x * wpb) {
    // owner rank and rank-local row of global row g
    const int b = a2a_seq_of(p.pad, B, g);
    const int pos = g - p.pad[b];
    const int cb = (p.pad[b + 1] - p.pad[b]) / (2 * cp);
    const int chunk = pos / cb;
    const int owner = chunk < cp ? chunk : 2 * cp - 1 - chunk;
    const int local = pos - chunk * cb + (chunk == owner ? 0 : cb);
    const int64_t srow = (int64_t)owner * rows_rank + p.pad[b] / cp + local;
#pragma unroll
    for (int j = 0; j < kA2aMaxJobs; ++j) {  // static indices keep the jobs in the parameter bank
      if (j >= p.njobs) break;
      const A2aJob& job = p.job[j];
      const int vph = p.D / 8;               // 16-byte vectors per head
      const int vpg = job.Hg * vph;          // per member
      const int nv = p.a2a * vpg;            // per token
      uint4* sh = reinterpret_cast<uint4*>(job.shard) + srow * nv;
      uint4* gr = reinterpret_cast<uint4*>(job.groups);
      const int64_t grow_stride = (int64_t)p.T * vpg;  // one member's tensor, in vectors
      for (int v0 = 0; v0 < nv; v0 += 32 * kA2aUnroll) {
        uint4 x[kA2aUnroll];
        int64_t goff[kA2aUnroll];
#pragma unroll
        for (int u = 0; u < kA2aUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          const int i = v / vpg;
          goff[u] = i * grow_stride + (int64_t)g * vpg + (v - i * vpg);
          if (v < nv) x[u] = kToGroups ? __ldg(sh + v) : __ldg(gr + goff[u]);
        }
#pragma unroll
        for (int u = 0; u < kA2aUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nv) {
            if (kToGroups) gr[goff[u]] = x[u];
            else sh[v] = x[u];
          }
        }
      }
    }
  }
}

cudaError_t launch_a2a(const A2aParams& p, bool to_groups, cudaStream_t st) {
  if (p.T == 0 || p.njobs == 0) return cudaSuccess;
  const int wpb = kA2aThreads / 32;
  const int64_t want = (p.T + wpb - 1) / wpb;
  const int grid = (int)(want < 8LL * num_sms() ? want : 8LL * num_sms());
  prof_before(THD_KERNEL_A2A, st);
  if (to_groups) a2a_kernel<true><<<grid, kA2aThreads, 0, st>>>(p);
  else a2a_kernel<false><<<grid, kA2aThreads, 0, st>>>(p);
  count_launch();
  cudaError_t e = cudaGetLastError();
  prof_after(THD_KERNEL_A2A, st);
  return e;
}

}  // namespace thd
