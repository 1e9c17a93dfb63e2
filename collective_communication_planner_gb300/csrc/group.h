// Internal state of a group and the host paths shared by the C ABI
// (api.cpp) and the copy-out engine's host side (copy_out_host.cpp).
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <memory>
#include <string>
#include <vector>

#include "internal.h"
#include "plan.h"
#include "reshard.h"
#include "tccl.h"

namespace tccl {

struct PlanKey {
  int coll;
  int elem_size;
  uint64_t count;
  int cap;
  std::string mod16;  // address mod 16 of every send then recv buffer
  int anchor = -1;    // >= 0: every window stores to this rank only (copy-out shard-in)
  int anchor_engine = 0;  // the engine of such a plan (bulk or TMA-reduce)
  bool in_place = false;
  bool operator<(const PlanKey& o) const {
    if (anchor != o.anchor) return anchor < o.anchor;
    if (anchor_engine != o.anchor_engine) return anchor_engine < o.anchor_engine;
    if (in_place != o.in_place) return o.in_place;
    if (coll != o.coll) return coll < o.coll;
    if (elem_size != o.elem_size) return elem_size < o.elem_size;
    if (count != o.count) return count < o.count;
    if (cap != o.cap) return cap < o.cap;
    return mod16 < o.mod16;
  }
};

struct CachedPlan {
  Lowered low;
  // bulk engine: one device allocation holding the window table, the chunk
  // prefix and the per-CTA scalar-window offsets
  unsigned char* d_table = nullptr;
  const Window* d_win = nullptr;
  const uint64_t* d_prefix = nullptr;
  const uint32_t* d_cta_first = nullptr;
  unsigned long long* d_sched = nullptr;
  // small engines: the launch argument block without its pointers
  std::vector<unsigned char> small_args;
  bool anchor_only = false;  // copy-out shard-in: the result goes to the anchor rank alone
  ~CachedPlan() {
    if (d_table) cudaFree(d_table);
  }
};

struct CachedReshard {
  ReshardPlan plan;
  unsigned char* d_table = nullptr;
  ~CachedReshard() {
    if (d_table) cudaFree(d_table);
  }
};

constexpr int kSmSlots = 64;
constexpr int kSmSlotWords = 8;  // 256 bits: one per SM

int log_level();  // TCCL_LOG: > 0 prints plans and launch errors to stderr
int elem_size_of(int dtype);
void fill_info(const Lowered& low, tcclLaunchInfo_t* info);

}  // namespace tccl

struct tcclGroup {
  int nranks = 0;
  int device = 0;
  tccl::DeviceDesc dev;
  tccl::Config cfg;
  int* d_status = nullptr;     // 64 bytes: [0] status code; bytes 32..47 the fused
                               // RMSNorm's row counter and finished-CTA count
  // SM recorder: one 256-bit bitmap per kernel launch while recording
  // (tccl::kSmSlots of them; launches past the last slot share it)
  uint32_t* d_sm_mask = nullptr;
  bool record_sms = false;
  int sm_launches = 0;         // launches recorded since the last read
  bool rms_cluster_enabled = true;  // TCCL_RMSNORM_CLUSTER=0 keeps one CTA per row
  uint64_t inject_ns = 0;
  std::map<tccl::PlanKey, std::unique_ptr<tccl::CachedPlan>> plans;
  std::map<std::string, std::unique_ptr<tccl::CachedReshard>> reshards;
  tcclLaunchInfo_t last;
  // copy-out engine: the group's own copy streams and the events that order
  // them after each segment's kernel and join them back to the caller
  std::vector<cudaStream_t> ce_streams;
  std::vector<cudaEvent_t> ce_seg_events;
  std::vector<cudaEvent_t> ce_done_events;
  cudaEvent_t ce_fork_event = nullptr;
};

namespace tccl {

// The SM bitmap the next kernel launch records into, or null when the group
// is not recording. Call once per launch.
inline uint32_t* sm_record_slot(tcclGroup* g) {
  if (!g->record_sms) return nullptr;
  const int slot = g->sm_launches < kSmSlots ? g->sm_launches : kSmSlots - 1;
  ++g->sm_launches;
  return g->d_sm_mask + (size_t)slot * kSmSlotWords;
}

// The plan (cached) of one call: its lowering and, for the bulk engines, its
// device tables. anchor >= 0: every window stores to that rank only (the
// copy-out engine's shard-in, on the bulk engine's TMA pipeline or, with
// anchor_engine = kEngineTmaReduce, on the TMA-reduce engine). A new plan's
// table upload is synchronous.
tcclResult_t get_plan(tcclGroup* g, int coll, const void* const* send, void* const* recv,
                      size_t count, int es, int cap, CachedPlan** out, int anchor = -1,
                      int anchor_engine = kEngineBulk);
// Launches one lowered plan on `stream`; returns a CUDA error code (0 on success).
int launch_plan(tcclGroup* g, CachedPlan* cp, int coll, int dtype, int op,
                const void* const* send, void* const* recv, int es, cudaStream_t stream);

// ---- copy-out engine (copy_out_host.cpp)
bool use_copy_out(const tcclGroup* g, int coll, size_t count, int es, int cap);
std::vector<uint8_t> mod16_of(int n, const void* const* p);
tcclResult_t run_copy_out_allreduce(tcclGroup* g, const void* const* send, void* const* recv,
                                    size_t count, int dtype, int op, int es, cudaStream_t stream,
                                    int cap);
tcclResult_t run_copy_out_reduce_scatter(tcclGroup* g, const void* const* send, void* const* recv,
                                         size_t rc, int dtype, int op, int es, cudaStream_t stream,
                                         int cap);
tcclResult_t run_copy_out_allgather(tcclGroup* g, const void* const* send, void* const* recv,
                                    size_t count, int es, cudaStream_t stream);

}  // namespace tccl
