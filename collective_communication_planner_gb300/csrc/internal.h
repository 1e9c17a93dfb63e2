// Internal types shared by the host planner/lowering (plan.cpp, api.cpp) and
// the device kernels (kernels.cu). Nothing here is part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

namespace tccl {

constexpr int kMaxRanks = 64;
constexpr int kSmallRanks = 8;    // small-argument class of the warp/vec engines
constexpr int kSmallWindows = 8;
constexpr int kLargeWindows = 3 * kMaxRanks + 2;

enum Coll : int { kAllReduce = 0, kReduceScatter = 1, kAllGather = 2 };
enum DType : int { kF32 = 0, kBF16 = 1, kI32 = 2 };
enum RedOp : int { kSum = 0, kMin = 1, kMax = 2 };
enum Engine : int {
  kEngineAuto = 0,
  kEngineBulk = 1,
  kEngineWarp = 2,
  kEngineVec = 3,
  kEngineTmaReduce = 4,
  kEngineCopyOut = 5  // bulk-engine shard-in to one anchor rank + copy-engine shard-out
};
enum StoreMode : int { kStoreAuto = 0, kStoreBulk = 1, kStoreVec = 2 };
enum ChunkOrder : int { kOrderAuto = 0, kOrderBlocked = 1, kOrderCyclic = 2, kOrderDynamic = 3 };
// Bulk engine stage layout: a stage holds one chunk of every source rank
// (kLayoutShared), or one rank's chunk (kLayoutPerRank: P stages per chunk,
// partial sums kept in registers, TMA copies as large as a whole stage).
enum StageLayout : int { kLayoutAuto = 0, kLayoutShared = 1, kLayoutPerRank = 2 };

constexpr int kMaxConsumerWarps = 16;  // bulk kernel: 1 + 16 warps = 544 threads
constexpr int kMaxReduceSlots = 8;     // TMA-reduce engine: chunk slots per issuing thread
// TMA-reduce engine: mbarriers (lanes x slots x buffers) its 1 KiB
// shared-memory head holds, beside a test barrier and the abort flag
constexpr int kReduceMaxBarriers = 120;
constexpr int kPerRankVectors = 4;     // per-rank layout: 16-byte vectors per consumer thread

// Status codes a kernel may leave in the group's status word (same values
// as tcclResult_t).
constexpr int kStatusTimeout = 4;

// One physical window: a contiguous byte range of a lowered task, resolved
// against the per-rank base pointers of the call. The "selected" source set
// is every rank's send buffer (src_sel < 0, a reduction) or one rank's
// (src_sel = r); likewise for destinations.
struct Window {
  uint64_t src_off;  // byte offset into each selected send buffer
  uint64_t dst_off;  // byte offset into each selected recv buffer
  uint32_t bytes;    // window length in bytes (multiple of the element size)
  int16_t src_sel;
  int16_t dst_sel;
  uint16_t scalar;   // 1: element-wise path (edge or not 16-byte co-aligned)
  uint16_t task;     // logical task (shard) the window came from
  int32_t cta;       // bulk engine scalar windows: owning CTA; otherwise -1
};
static_assert(sizeof(Window) == 32, "Window layout");

template <int MAXR>
struct BasePtrs {
  const void* src[MAXR];
  void* dst[MAXR];
};

// Bulk (TMA pipeline) engine. The plan's body windows (16-byte co-aligned)
// form one sequence of equal chunks (each window's last chunk may be short).
// CTA j takes the range [j*k, (j+1)*k) (blocked order), chunks j, j+G, j+2G,
// ... (cyclic order: all CTAs sweep the buffers together), or claims chunks
// one at a time from a device counter (dynamic order: faster SMs take more).
// Element-wise windows are bound to CTAs.
struct BulkArgs {
  BasePtrs<kMaxRanks> p;
  const Window* win;             // device table: nbody body windows, then scalar windows
  const uint64_t* chunk_prefix;  // device table, nbody + 1 entries: chunks before body window w
  const uint32_t* cta_first;     // device table, grid + 1 entries: CTA j's scalar windows are
                                 // win[nbody + cta_first[j] .. nbody + cta_first[j + 1])
  int* status;                   // status word (device)
  uint32_t* sm_mask;             // SM recorder bitmap (device) or null
  uint64_t timeout_ns;           // bound on every wait
  uint64_t inject_timeout_ns;    // test hook: > 0 makes CTA 0 wait on a barrier nothing signals
  uint64_t total_chunks;
  uint64_t chunks_per_cta;       // blocked order
  unsigned long long* sched;     // dynamic order: {next chunk, CTAs finished}, zero between launches
  int nbody;
  int order;                     // kOrderBlocked, kOrderCyclic or kOrderDynamic
  int nranks;
  int chunk_bytes;               // bytes per source per chunk (multiple of 16)
  int stages;
  int store_mode;                // kStoreBulk or kStoreVec
  int consumer_warps;
  int release_lag;               // all-gather bulk stores: store groups kept in flight
  int elem_size;
  int rank_streamed;             // kLayoutPerRank (1) or kLayoutShared (0)
  int prefetch_chunks;           // L2 prefetch distance beyond the shared-memory ring (0: off)
  int load_evict_first;          // bulk loads carry an L2 evict-first policy
  int arrival_order;             // TMA-reduce engine: ranks 1..P-1 reduced as they arrive
  int reduce_slots;              // TMA-reduce engine: chunks each issuing thread keeps in flight
  int reduce_bufs;               // TMA-reduce engine: buffers per slot (2, or 3 for reduce-scatter)
  int anchor_only;               // TMA-reduce engine: allreduce into the anchor only (no shard-out)
};

// Warp / vec (small-message) engines: the whole lowered plan rides in the
// kernel parameters, so a launch reads no table from memory.
template <int MAXR, int MAXW>
struct SmallArgs {
  BasePtrs<MAXR> p;
  Window win[MAXW];
  uint64_t vec_prefix[MAXW + 1];   // 16-byte units before window w (vector windows only)
  uint64_t elem_prefix[MAXW + 1];  // elements before window w (scalar windows only)
  uint32_t* sm_mask;
  int nwin;
  int nranks;
  int elem_size;
};

struct LaunchShape {
  int engine = 0;
  int store_mode = 0;
  int grid = 0;
  int threads = 0;
  int stages = 0;
  int chunk_bytes = 0;
  int consumer_warps = 0;
  int release_lag = 0;
  int order = 0;
  int rank_streamed = 0;
  int prefetch_chunks = 0;
  int load_evict_first = 0;
  int early_launch = 0;  // bulk engine, uncapped: programmatic dependent launch
  int reduce_slots = 0;  // TMA-reduce engine: chunk slots per issuing thread
  int reduce_bufs = 0;   // TMA-reduce engine: buffers per slot
  size_t smem = 0;
};

// Kernel launchers (kernels.cu). Each returns a cudaError_t as int.
int launch_bulk(int coll, int dtype, int op, const BulkArgs& a, const LaunchShape& s,
                void* stream);
int launch_small_ar(int dtype, int op, int engine, int size_class, const void* args,
                    const LaunchShape& s, void* stream);
int launch_small_rs(int dtype, int op, int engine, int size_class, const void* args,
                    const LaunchShape& s, void* stream);
int launch_small_ag(int dtype, int op, int engine, int size_class, const void* args,
                    const LaunchShape& s, void* stream);
int launch_reduce(int coll, int dtype, int op, const BulkArgs& a, const LaunchShape& s,
                  void* stream);
// (dtype, op) pairs the copy hardware reduces exactly in a fixed order
inline bool tma_reduce_supported(int dtype, int op) {
  return (dtype == kF32 && op == kSum) || dtype == kI32 || (dtype == kBF16 && op != kSum);
}
int prepare_bulk_kernels(size_t smem_bytes);  // opt-in shared memory for the bulk kernels

}  // namespace tccl
