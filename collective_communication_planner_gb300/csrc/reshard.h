// M-to-N reshard planner (host only).
//
// Follows the M2N part of the "NCCL M2N vs T-CCL" article (§1.2-§1.4): a
// layout is a mesh of ranks (row-major, contiguous from a base rank) with one
// placement per mesh axis, Shard(d) or Replicate(), at most one sharded axis.
// The plan is derived from the layouts alone by interval intersection: each
// destination block receives exactly the bytes it needs, each source block
// feeding it is read once (from a source replica chosen so that replicas'
// loads differ by at most one) and written to every destination replica of
// that block (the article's leader + in-domain fan-out, which on one GPU is
// "load once, store to all").
#pragma once

#include <string>
#include <vector>

#include "internal.h"

namespace tccl {

constexpr int kMaxMeshDims = 4;
constexpr int kMaxTensorDims = 4;
constexpr int kReplicate = -1;

struct MeshLayout {
  int ndims = 0;
  int dims[kMaxMeshDims] = {0, 0, 0, 0};
  int start = 0;
  int place[kMaxMeshDims] = {kReplicate, kReplicate, kReplicate, kReplicate};
  int size() const {
    int n = 1;
    for (int i = 0; i < ndims; ++i) n *= dims[i];
    return n;
  }
};

struct Box {
  uint64_t lo[kMaxTensorDims];
  uint64_t hi[kMaxTensorDims];
};

// One strided copy: `nrows` rows of `bytes`, from one source rank's buffer to
// every destination rank in `dst_mask` (all replicas of one block, same
// offsets). 64 bytes.
struct ReshardWindow {
  uint64_t src_off;
  uint64_t dst_off;
  uint64_t src_pitch;
  uint64_t dst_pitch;
  uint64_t dst_mask;
  uint32_t bytes;
  uint32_t nrows;
  uint32_t src;     // source mesh rank
  uint32_t scalar;  // 1: element-wise path (not 16-byte co-aligned)
  uint32_t pad[2];
};
static_assert(sizeof(ReshardWindow) == 64, "ReshardWindow layout");

struct ReshardTransfer {  // logical: one source block part to one destination block
  int src_rank;            // chosen source mesh rank
  uint64_t dst_mask;       // destination replicas
  Box box;                 // global coordinates
};

// How a plan's copies run.
enum ReshardEngine : int {
  kReshardWarp = 0,  // warps copy row segments through registers (any alignment)
  kReshardBulk = 1,  // a shared-memory ring per CTA: bulk loads in, bulk stores out
};

struct ReshardPlan {
  std::vector<ReshardTransfer> transfers;
  std::vector<ReshardWindow> win;
  std::vector<uint64_t> unit_prefix;  // work units before window w (nwin + 1 entries)
  std::vector<int> src_load;          // transfers read from each source mesh rank
  uint64_t bytes_read = 0;
  uint64_t bytes_written = 0;
  int engine = kReshardWarp;
  int grid = 0;
  int threads = 0;
  size_t smem = 0;  // dynamic shared memory per CTA
};

// Validates a layout against the tensor (returns false with a reason).
bool check_layout(const MeshLayout& l, int nd, const uint64_t* shape, std::string* why);

// Global box held by mesh rank m of layout l.
Box layout_box(const MeshLayout& l, int nd, const uint64_t* shape, int m);

// Plans and lowers one reshard. src_mod16 / dst_mod16: each rank's buffer
// address mod 16. engine (the group's tcclEngine_t setting): Warp or Vec keep
// the copies on the warp kernel; Bulk puts them on the bulk ring whenever
// every window is 16-byte co-aligned and a ring fits in smem_per_block bytes
// of shared memory; Auto (and any other) does so only where the ring was
// measured faster: every block written to kReshardBulkMinFanout or more
// replicas on average and every row piece of kReshardBulkMinRowBytes or more.
// Returns false with a reason on an invalid request.
bool plan_reshard(const MeshLayout& src, const MeshLayout& dst, int nd, const uint64_t* shape,
                  int elem_size, const uint8_t* src_mod16, const uint8_t* dst_mod16,
                  int sm_count, int cta_cap, int engine, size_t smem_per_block,
                  ReshardPlan* out, std::string* why);

// A warp work unit is one segment of one row: up to kReshardSegBytes of a
// vector window, or up to kReshardSegElems elements of a scalar window.
constexpr uint32_t kReshardSegBytes = 4096;
constexpr uint32_t kReshardSegElems = 1024;

// Bulk engine: one CTA per SM (within the cap) with a ring of
// kReshardBulkStages stages of kReshardBulkSegBytes. A work unit is one
// stage's worth: a segment of a row longer than a stage, or as many whole
// rows of a shorter one as fit. One thread issues the unit's bulk loads,
// another its bulk stores to every destination replica.
constexpr uint32_t kReshardBulkSegBytes = 16384;
constexpr int kReshardBulkStages = 8;
// stages held by stores before a stage is freed: half the ring, which keeps
// the bytes in flight split as the traffic is (1 read to fan-out writes)
constexpr int kReshardBulkLag = kReshardBulkStages / 2;
constexpr uint64_t kReshardBulkMinFanout = 3;
constexpr uint32_t kReshardBulkMinRowBytes = 4096;
constexpr int kReshardBulkThreads = 64;
constexpr size_t kReshardBulkHeadBytes = 1024;  // barriers, stage descriptors

// Units of a vector window on the bulk engine, and what unit k covers: rows
// [row, row + rows) and bytes [begin, begin + n) of each.
struct BulkUnit {
  uint32_t row, rows, begin, n;
};
inline uint64_t bulk_units(uint32_t bytes, uint32_t nrows) {
  if (bytes >= kReshardBulkSegBytes)
    return (uint64_t)nrows * ((bytes + kReshardBulkSegBytes - 1) / kReshardBulkSegBytes);
  const uint32_t per = kReshardBulkSegBytes / bytes;
  return ((uint64_t)nrows + per - 1) / per;
}

struct ReshardArgs {
  const ReshardWindow* win;
  const uint64_t* unit_prefix;
  unsigned long long* sched;  // bulk engine: two zeroed claim words of this plan
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  uint32_t* sm_mask;
  int* status;            // bulk engine: the group's status word (a wait ran out)
  uint64_t timeout_ns;    // bulk engine: bound on every wait
  uint64_t inject_timeout_ns;  // test hook: CTA 0's first stage waits this long on a barrier nothing completes
  int nwin;
  int elem_size;
};

// early: programmatic dependent launch (uncapped calls only)
int launch_reshard(const ReshardArgs& a, int grid, bool early, void* stream);
int launch_reshard_bulk(const ReshardArgs& a, int grid, size_t smem, bool early, void* stream);
// opt-in shared memory for the bulk engine's ring (once per device)
int prepare_reshard_kernels(size_t smem_bytes);

}  // namespace tccl
