// Copy-out engine: the shard-in kernel that folds P ranks into one anchor
// rank's buffer with plain 128-bit register loads (no shared-memory staging),
// before the GPU's copy engines fan the result out to the other ranks.
#pragma once

#include "internal.h"

namespace tccl {

constexpr int kAnchorThreads = 1024;
constexpr uint64_t kAnchorMaxVectors = (uint64_t)1 << 28;  // per launch (4 GiB per rank)

// One segment of a copy-out allreduce. All P sources and the destination
// share their address mod 16: `head_bytes` element-wise bytes, then `nvec`
// 16-byte vectors, then `tail_bytes` element-wise bytes.
struct AnchorArgs {
  BasePtrs<kMaxRanks> p;  // p.src[0..P-1] the sends, p.dst[0] the anchor's receive buffer
  uint32_t* sm_mask;      // SM recorder bitmap or null
  uint64_t head_bytes;
  uint64_t nvec;
  uint64_t tail_bytes;
  int nranks;
};

// `vectors_per_thread` is 1 or 2 (loads in flight per thread: 8 either way).
int launch_anchor_reduce(int dtype, int op, const AnchorArgs& a, int grid, int vectors_per_thread,
                         void* stream);

}  // namespace tccl
