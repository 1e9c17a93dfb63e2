// Allreduce fused with RMSNorm: launch arguments and limits.
#pragma once

#include "internal.h"

namespace tccl {

constexpr int kRmsMaxThreads = 256;
constexpr int kRmsMaxVectors = 8;  // 16-byte vectors of a row per thread

struct RmsArgs {
  BasePtrs<kMaxRanks> p;
  const void* gamma;  // hidden elements, the output type
  uint32_t* sm_mask;
  uint64_t rows;
  uint32_t hidden;
  float eps;
  int nranks;
};

// `vectors`: 16-byte vectors of a row per thread (4 or 8); gamma is staged in
// hidden * element-size bytes of dynamic shared memory.
int launch_rmsnorm(int dtype, const RmsArgs& a, int grid, int threads, int vectors, void* stream);

}  // namespace tccl
