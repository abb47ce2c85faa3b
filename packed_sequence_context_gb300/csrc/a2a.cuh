// Parameters of the emulated all-to-all (a2a.cu): the layouts it moves
// between are described there.
#pragma once
#include "common.cuh"

namespace thd {

// One tensor to move: its shard buffer [cp][T/cp, a2a * Hg, D] and its
// per-member buffer [a2a][T, Hg, D] (bf16; D a multiple of 8).
struct A2aJob {
  void* shard;
  void* groups;
  int Hg;  // heads per member
};

constexpr int kA2aMaxJobs = 5;

struct A2aParams {
  A2aJob job[kA2aMaxJobs];
  int njobs;
  const int32_t* pad;  // cu_seqlens_padded [B+1], validated by the planner
  const int32_t* dev_status;
  int B, cp, a2a, D;
  int64_t T;  // shard stride is T / cp rows; rows past pad[B] are not moved
};

// to_groups: shards -> per-member buffers (the A2A in front of attention);
// otherwise per-member buffers -> shards (the A2A behind it).
cudaError_t launch_a2a(const A2aParams& p, bool to_groups, cudaStream_t st);

}  // namespace thd
