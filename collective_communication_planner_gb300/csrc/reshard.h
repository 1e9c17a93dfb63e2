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

struct ReshardPlan {
  std::vector<ReshardTransfer> transfers;
  std::vector<ReshardWindow> win;
  std::vector<uint64_t> unit_prefix;  // warp work units before window w (nwin + 1 entries)
  std::vector<int> src_load;          // transfers read from each source mesh rank
  uint64_t bytes_read = 0;
  uint64_t bytes_written = 0;
  int grid = 0;
};

// Validates a layout against the tensor (returns false with a reason).
bool check_layout(const MeshLayout& l, int nd, const uint64_t* shape, std::string* why);

// Global box held by mesh rank m of layout l.
Box layout_box(const MeshLayout& l, int nd, const uint64_t* shape, int m);

// Plans and lowers one reshard. src_mod16 / dst_mod16: each rank's buffer
// address mod 16. Returns false with a reason on an invalid request.
bool plan_reshard(const MeshLayout& src, const MeshLayout& dst, int nd, const uint64_t* shape,
                  int elem_size, const uint8_t* src_mod16, const uint8_t* dst_mod16,
                  int sm_count, int cta_cap, ReshardPlan* out, std::string* why);

// A warp work unit is one segment of one row: up to kReshardSegBytes of a
// vector window, or up to kReshardSegElems elements of a scalar window.
constexpr uint32_t kReshardSegBytes = 4096;
constexpr uint32_t kReshardSegElems = 1024;

struct ReshardArgs {
  const ReshardWindow* win;
  const uint64_t* unit_prefix;
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  uint32_t* sm_mask;
  int nwin;
  int elem_size;
};

// early: programmatic dependent launch (uncapped calls only)
int launch_reshard(const ReshardArgs& a, int grid, bool early, void* stream);

}  // namespace tccl
