// Task planner and lowering pass (host only).
//
// The planner follows T-CCL's task-based planning ("NCCL M2N vs T-CCL"
// article, section 2.3): the logical tensor is split into P shards, shard s
// is owned by rank s, and the planner emits logical tasks {op, executing
// rank, source intervals, destination intervals, dependencies}. The lowering
// pass resolves each logical task into physical ones (addresses relative to
// the call's base pointers, and the transfer mechanism), then cuts them into
// windows and chunks for one engine (same section, "lower" and "TMA engine").
#pragma once

#include <string>
#include <vector>

#include "internal.h"

namespace tccl {

// Element interval [begin, end) of one rank's buffer.
struct Interval {
  int rank;
  uint64_t begin;
  uint64_t end;
};

enum TaskKind : int {
  kShardIn = 0,   // load every rank's part of the shard and reduce it at the owner
  kShardOut = 1,  // take the owner's final shard once and store it to every rank
};

// Where a task's intervals live.
enum BufKind : int { kSendBuf = 0, kRecvBuf = 1, kOwnerShard = 2 };

struct LogicalTask {
  TaskKind kind;
  int op;           // reduction (shard-in) or -1 (shard-out copies)
  int exec_rank;    // the shard's owner
  int shard;
  BufKind src_buf;
  BufKind dst_buf;
  std::vector<Interval> src;
  std::vector<Interval> dst;
  std::vector<int> deps;  // indices of tasks that must finish first
};

struct Plan {
  int coll = 0;
  int nranks = 0;
  int elem_size = 0;
  int op = 0;
  uint64_t count = 0;        // the call's count argument
  uint64_t shard_elems = 0;  // shard length q
  std::vector<LogicalTask> tasks;
  // facts about the call that steer the lowering (not part of the tasks)
  bool in_place = false;     // allreduce: every rank's receive buffer is its send buffer
  bool anchor_only = false;  // every window will store to one rank only (copy-out shard-in)
};

// Splits the collective into logical tasks.
Plan plan_collective(int coll, int nranks, uint64_t count, int elem_size, int op);

struct DeviceDesc {
  int sm_count = 0;
  int smem_optin = 0;   // max dynamic shared memory per block (opt-in)
  int smem_per_sm = 0;  // shared memory per SM
};

struct Config {
  int engine = kEngineAuto;
  size_t small_max_bytes = 0;
  size_t vec_max_bytes = 0;
  int stage_bytes = 0;
  int stages = 0;
  int store_mode = kStoreAuto;
  int consumer_warps = 0;
  int ctas_per_sm = 0;
  double wait_timeout_ms = 0;
  int chunk_order = kOrderAuto;
  int stage_layout = kLayoutAuto;
  int prefetch_chunks = -1;   // -1: library default
  int load_policy = 0;        // 0 default (evict-normal), 1 evict-first, 2 evict-normal
  size_t max_chunk_bytes = 0;
  int ce_streams = 0;
  size_t ce_segment_bytes = 0;
  int ce_auto_max_cap = 0;
  int reduce_order = 0;  // 0 ascending, 1 arrival (TMA-reduce engine only)
  int ce_fold = 0;       // copy-out allreduce shard-in: kFoldAuto / kFoldRegister / kFoldTma
  int ce_tail_percent = 0;  // copy-out allreduce: last segment's length, % of the others (0: 100)
  int reduce_slots = 0;     // TMA-reduce engine: chunks each issuing thread keeps in flight (0: default)
  int ce_ar_streams = 0;    // copy-out allreduce: copy streams of each segment but the last (0: by cap)
  int ce_tail_streams = 0;  // copy-out allreduce: copy streams of the last segment
};

// The copy-out allreduce's shard-in kernel. Auto and Register: the
// register-load fold wherever the buffers allow it (register_fold_ok), else
// the bulk engine's TMA pipeline; Tma: always the TMA pipeline; TmaReduce:
// the TMA-reduce engine into the anchor (the copy hardware reduces, no thread
// touches the data), for the (dtype, op) pairs it reduces exactly, else Auto.
enum CeFold : int { kFoldAuto = 0, kFoldRegister = 1, kFoldTma = 2, kFoldTmaReduce = 3 };

// Fills zero fields with the library defaults (small_max_bytes stays 0: it
// depends on the rank count, see small_max_bytes()).
Config resolve_config(const Config& in);

// The largest message per rank buffer Auto gives the warp engine: the
// config's small_max_bytes, or when that is 0, 64 KiB for P >= 5 and 128 KiB
// below.
uint64_t small_max_bytes(const Config& c, int nranks);

// Up to this many lanes per SM the vec engine spreads its lanes over one CTA
// per SM (CTAs of the lanes / SMs, rounded up to a warp); above, CTAs of 256.
constexpr uint64_t kVecSpreadLanesPerSm = 192;

// The bulk engine's default pipeline shape. With all three at these values
// an uncapped, out-of-place allreduce that stores to every rank and moves at
// least kArInflightMinTraffic bytes (2 * P * S) sizes its ring for
// kArInflightBytes of loads in flight per CTA (chunks of at least
// kArMinChunkBytes); other calls, and any shape set explicitly, use
// stage_bytes / stages / max_chunk_bytes as given (stages reduced to what
// shared memory holds).
constexpr int kDefaultStageBytes = 64 * 1024;
constexpr int kDefaultStages = 8;
constexpr size_t kDefaultMaxChunkBytes = 16384;
constexpr uint64_t kArInflightBytes = 96 * 1024;
constexpr uint64_t kArMinChunkBytes = 6144;
constexpr uint64_t kArInflightMinTraffic = (uint64_t)512 << 20;
// TMA-reduce engine defaults (max_chunk_bytes left at its default selects
// kDefaultReduceChunkBytes)
constexpr int kDefaultReduceSlots = 4;
constexpr uint64_t kDefaultReduceChunkBytes = 8192;
inline bool default_bulk_shape(const Config& c) {
  return c.stage_bytes == kDefaultStageBytes && c.stages == kDefaultStages &&
         c.max_chunk_bytes == kDefaultMaxChunkBytes;
}

// ---- copy-out engine decisions (host only; the launches and copies live in
// copy_out_host.cpp, the fold kernel in kernels_copy_out.cu)
constexpr int kMaxCeSegments = 64;
constexpr size_t kCeAutoMinBytes = (size_t)4 << 20;
constexpr uint64_t kFoldMaxVectors = (uint64_t)1 << 28;  // per launch job, 32-bit indices

// Whether a call runs on the copy-out engine: always when the group's engine
// is copy-out (P >= 2); under Auto, for calls of at least 4 MiB per rank
// buffer (allreduce: the buffer; reduce-scatter: the send buffer; all-gather:
// the receive buffer): allreduce / all-gather when 0 < cap <= ce_auto_max_cap
// (default by P, copy_out_auto_max_cap), reduce-scatter under any cap or uncapped with
// P <= 4. ce_auto_max_cap < 0 turns Auto's choice off.
bool copy_out_chosen(const Config& c, int sm_count, int nranks, int coll, size_t count, int es,
                     int cap);

// The largest cap for which Auto picks the copy-out engine for an allreduce
// or all-gather: ce_auto_max_cap when set, else 4/7 of the SMs for P <= 2,
// 5/12 for P = 3 and 4, 7/16 for P >= 5 (86, 63 and 66 on 152 SMs).
int copy_out_auto_max_cap(const Config& c, int sm_count, int nranks);

// Segments of a copy-out allreduce of `count` elements: at most
// ce_segment_bytes per rank, at least four where each stays >= 4 MiB, at most
// kMaxCeSegments, offsets multiples of 256 bytes. *seg_elems is the length of
// every segment but the last (which holds the rest). With ce_tail_percent
// below 100, the same number of segments is kept and the last one is cut to
// about that share of the others, which grow (past ce_segment_bytes if need
// be) to cover the rest: the last segment's copies overlap no fold, so a
// shorter last segment shortens the call's exposed tail.
void copy_out_segments(const Config& c, size_t count, int es, size_t* seg_elems, int* nseg);

// Whether the register-load fold takes a copy-out call (else the TMA
// pipeline, or for reduce-scatter the bulk engine): every send buffer shares
// its address mod 16 with the receive buffer(s) written (allreduce: rank 0's;
// reduce-scatter: every rank's, and a shard must be a multiple of 16 bytes),
// and a launch job stays below kFoldMaxVectors vectors. `seg_elems` is the
// allreduce's segment length (ignored for reduce-scatter).
bool register_fold_ok(int coll, int nranks, const uint8_t* send_mod16, const uint8_t* recv_mod16,
                      size_t count, int es, size_t seg_elems);

// Copy streams of a copy-out allreduce: *mid for the segments whose copies
// run beside the next segment's fold (ce_ar_streams, or by default one per
// 112 / (P - 1) CTAs of the cap, rounded, at least 1: one per 16 CTAs for
// P = 8), *tail for the last segment
// (ce_tail_streams); both within ce_streams and P - 1.
void copy_out_streams(const Config& c, int nranks, int cap, int* mid, int* tail);

// Whether a copy-out allreduce's segments fold with the register-load kernel
// (else the TMA pipeline): register_fold_ok, unless the config asks for the
// TMA pipeline (ce_fold = kFoldTma).
bool allreduce_register_fold(const Config& c, int nranks, const uint8_t* send_mod16,
                             const uint8_t* recv_mod16, size_t count, int es, size_t seg_elems);

struct Lowered {
  LaunchShape shape;
  std::vector<Window> win;           // bulk: body windows, then scalar windows by CTA;
                                     // small engines: in plan order
  int nbody = 0;                     // bulk: body windows at the front of `win`
  std::vector<uint64_t> chunk_prefix;  // bulk: nbody + 1 entries
  uint64_t total_chunks = 0;         // bulk
  uint64_t chunks_per_cta = 0;       // bulk, blocked order
  std::vector<uint32_t> cta_first;   // bulk: grid + 1 entries into the scalar windows
  std::vector<uint64_t> vec_prefix;  // small engines: nwin + 1 entries
  std::vector<uint64_t> elem_prefix; // small engines: nwin + 1 entries
  int ntasks = 0;
  int size_class = 0;  // small engines: 0 = (8 ranks, 8 windows), 1 = (64, 194)
};

// Lowers a plan for the given buffer alignments (address mod 16 of each
// rank's send and recv buffer). Returns false with a reason when the
// configuration cannot be lowered (which the API reports as invalid usage).
bool lower_plan(const Plan& plan, const uint8_t* send_mod16, const uint8_t* recv_mod16,
                const Config& cfg, const DeviceDesc& dev, int cta_cap, Lowered* out,
                std::string* why);

// Serialises a bulk plan's device table: windows, then the chunk prefix
// (8-byte aligned), then the per-CTA scalar-window offsets, then the two
// zeroed scheduler words of the dynamic chunk order.
void pack_bulk_table(const Lowered& low, std::vector<unsigned char>* out, size_t* off_prefix,
                     size_t* off_cta, size_t* off_sched);

// Checks a collective call's arguments: enums, rank count, null and
// misaligned pointers, size overflow, and buffer overlap (only the NCCL
// in-place forms may alias). Returns a tcclResult_t value.
int validate_collective_args(int coll, int nranks, const void* const* send, void* const* recv,
                             size_t count, int dtype, int op);

// [a, a + na) and [b, b + nb) share a byte.
bool ranges_overlap(uintptr_t a, size_t na, uintptr_t b, size_t nb);

// Per-rank message size the Auto engine choice looks at.
uint64_t message_bytes(int coll, int nranks, uint64_t count, int elem_size);

}  // namespace tccl
