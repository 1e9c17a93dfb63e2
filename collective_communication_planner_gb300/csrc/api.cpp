// C ABI of the library (include/tccl.h): argument validation, the plan
// cache, device tables and launches. Host code only; kernels live in the .cu
// translation units.
#include "tccl.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <string>
#include <vector>

#include "copy_out.h"
#include "group.h"
#include "internal.h"
#include "plan.h"
#include "reshard.h"
#include "rmsnorm.h"

using namespace tccl;

namespace tccl {

namespace {
int elem_size_of_dtype(int dtype) { return dtype == kBF16 ? 2 : 4; }
}  // namespace

bool ranges_overlap(uintptr_t a, size_t na, uintptr_t b, size_t nb) {
  if (na == 0 || nb == 0) return false;
  return a < b + nb && b < a + na;
}

// Argument rules shared by every collective entry point (see plan.h).
int validate_collective_args(int coll, int nranks, const void* const* send, void* const* recv,
                             size_t count, int dtype, int op) {
  if (coll < kAllReduce || coll > kAllGather) return tcclInvalidArgument;
  if (nranks < 1 || nranks > TCCL_MAX_RANKS) return tcclInvalidArgument;
  if (dtype < kF32 || dtype > kI32) return tcclInvalidArgument;
  if (coll != kAllGather && (op < kSum || op > kMax)) return tcclInvalidArgument;
  if (!send || !recv) return tcclInvalidArgument;
  if (count == 0) return tcclSuccess;
  const int es = elem_size_of_dtype(dtype);
  const uint64_t big = (uint64_t)nranks * (uint64_t)es;
  if (count > (SIZE_MAX / 4) / big) return tcclInvalidArgument;
  const size_t sbytes = (coll == kReduceScatter ? nranks * count : count) * es;
  const size_t rbytes = (coll == kAllGather ? nranks * count : count) * es;
  const size_t shard_bytes = count * es;
  for (int r = 0; r < nranks; ++r) {
    if (!send[r] || !recv[r]) return tcclInvalidArgument;
    if (((uintptr_t)send[r] % es) || ((uintptr_t)recv[r] % es)) return tcclInvalidArgument;
  }
  for (int r = 0; r < nranks; ++r) {
    const uintptr_t rr = (uintptr_t)recv[r];
    const uintptr_t sr = (uintptr_t)send[r];
    // the recv buffer against its own rank's send buffer: in place the NCCL
    // way, or disjoint
    bool in_place = false;
    if (coll == kAllReduce) in_place = (rr == sr);
    if (coll == kReduceScatter) in_place = (rr == sr + r * shard_bytes);
    if (coll == kAllGather) in_place = (sr == rr + r * shard_bytes);
    if (!in_place && ranges_overlap(rr, rbytes, sr, sbytes)) return tcclInvalidArgument;
    for (int k = 0; k < nranks; ++k) {
      if (k == r) continue;
      if (ranges_overlap(rr, rbytes, (uintptr_t)recv[k], rbytes)) return tcclInvalidArgument;
      if (ranges_overlap(rr, rbytes, (uintptr_t)send[k], sbytes)) return tcclInvalidArgument;
    }
  }
  return tcclSuccess;
}

}  // namespace tccl

namespace {

template <int MAXR, int MAXW>
void build_small_args(const Lowered& low, int nranks, int elem_size,
                      std::vector<unsigned char>* out) {
  out->assign(sizeof(SmallArgs<MAXR, MAXW>), 0);
  auto* a = reinterpret_cast<SmallArgs<MAXR, MAXW>*>(out->data());
  a->nwin = (int)low.win.size();
  a->nranks = nranks;
  a->elem_size = elem_size;
  for (size_t i = 0; i < low.win.size(); ++i) a->win[i] = low.win[i];
  for (size_t i = 0; i < low.vec_prefix.size(); ++i) {
    a->vec_prefix[i] = low.vec_prefix[i];
    a->elem_prefix[i] = low.elem_prefix[i];
  }
}

template <int MAXR, int MAXW>
void fill_small_ptrs(std::vector<unsigned char>* buf, int nranks, const void* const* send,
                     void* const* recv, uint32_t* sm_mask) {
  auto* a = reinterpret_cast<SmallArgs<MAXR, MAXW>*>(buf->data());
  for (int r = 0; r < nranks; ++r) {
    a->p.src[r] = send[r];
    a->p.dst[r] = recv[r];
  }
  a->sm_mask = sm_mask;
}

// Nothing to move: one rank, in place.
bool is_noop(int coll, int nranks, const void* const* send, void* const* recv) {
  if (nranks != 1) return false;
  (void)coll;
  return send[0] == recv[0];
}

Config config_from_env() {
  Config c;
  auto geti = [](const char* n, int d) {
    const char* e = std::getenv(n);
    return e ? std::atoi(e) : d;
  };
  if (const char* e = std::getenv("TCCL_ENGINE")) {
    std::string v(e);
    if (v == "tma_reduce") c.engine = kEngineTmaReduce;
    if (v == "bulk") c.engine = kEngineBulk;
    else if (v == "warp") c.engine = kEngineWarp;
    else if (v == "vec") c.engine = kEngineVec;
    else if (v == "copy_out") c.engine = kEngineCopyOut;
  }
  c.ce_streams = geti("TCCL_CE_STREAMS", 0);
  if (const char* e = std::getenv("TCCL_CE_SEGMENT_BYTES")) c.ce_segment_bytes = std::strtoull(e, 0, 10);
  c.ce_auto_max_cap = geti("TCCL_CE_AUTO_MAX_CAP", 0);
  if (const char* e = std::getenv("TCCL_REDUCE_ORDER")) c.reduce_order = std::string(e) == "arrival" ? 1 : 0;
  c.ce_tail_percent = geti("TCCL_CE_TAIL_PERCENT", 0);
  c.reduce_slots = geti("TCCL_REDUCE_SLOTS", 0);
  c.ce_ar_streams = geti("TCCL_CE_AR_STREAMS", 0);
  c.ce_tail_streams = geti("TCCL_CE_TAIL_STREAMS", 0);
  if (const char* e = std::getenv("TCCL_CE_FOLD")) {
    std::string v(e);
    if (v == "register") c.ce_fold = kFoldRegister;
    else if (v == "tma") c.ce_fold = kFoldTma;
  }
  if (const char* e = std::getenv("TCCL_SMALL_MAX_BYTES")) c.small_max_bytes = std::strtoull(e, 0, 10);
  if (const char* e = std::getenv("TCCL_VEC_MAX_BYTES")) c.vec_max_bytes = std::strtoull(e, 0, 10);
  c.stage_bytes = geti("TCCL_STAGE_BYTES", 0);
  c.stages = geti("TCCL_STAGES", 0);
  if (const char* e = std::getenv("TCCL_STORE_MODE")) {
    std::string v(e);
    if (v == "bulk") c.store_mode = kStoreBulk;
    else if (v == "vec") c.store_mode = kStoreVec;
  }
  c.consumer_warps = geti("TCCL_CONSUMER_WARPS", 0);
  c.prefetch_chunks = geti("TCCL_PREFETCH_CHUNKS", -1);
  c.load_policy = geti("TCCL_LOAD_POLICY", 0);
  if (const char* e = std::getenv("TCCL_MAX_CHUNK_BYTES")) c.max_chunk_bytes = std::strtoull(e, 0, 10);
  if (const char* e = std::getenv("TCCL_STAGE_LAYOUT")) {
    std::string v(e);
    if (v == "shared") c.stage_layout = kLayoutShared;
    else if (v == "per_rank") c.stage_layout = kLayoutPerRank;
  }
  if (const char* e = std::getenv("TCCL_CHUNK_ORDER")) {
    std::string v(e);
    if (v == "blocked") c.chunk_order = kOrderBlocked;
    else if (v == "cyclic") c.chunk_order = kOrderCyclic;
    else if (v == "dynamic") c.chunk_order = kOrderDynamic;
  }
  c.ctas_per_sm = geti("TCCL_CTAS_PER_SM", 0);
  if (const char* e = std::getenv("TCCL_WAIT_TIMEOUT_MS")) c.wait_timeout_ms = std::atof(e);
  return resolve_config(c);
}

Config from_public(const tcclConfig_t& p) {
  Config c;
  c.engine = p.engine;
  c.small_max_bytes = p.small_max_bytes;
  c.vec_max_bytes = p.vec_max_bytes;
  c.stage_bytes = p.stage_bytes;
  c.stages = p.stages;
  c.store_mode = p.store_mode;
  c.consumer_warps = p.consumer_warps;
  c.ctas_per_sm = p.ctas_per_sm;
  c.wait_timeout_ms = p.wait_timeout_ms;
  c.chunk_order = p.chunk_order;
  c.stage_layout = p.stage_layout;
  c.prefetch_chunks = p.prefetch_chunks;
  c.load_policy = p.load_policy;
  c.max_chunk_bytes = p.max_chunk_bytes;
  c.ce_streams = p.ce_streams;
  c.ce_segment_bytes = p.ce_segment_bytes;
  c.ce_auto_max_cap = p.ce_auto_max_cap;
  c.reduce_order = p.reduce_order;
  c.ce_fold = p.ce_fold;
  c.ce_tail_percent = p.ce_tail_percent;
  c.reduce_slots = p.reduce_slots;
  c.ce_ar_streams = p.ce_ar_streams;
  c.ce_tail_streams = p.ce_tail_streams;
  return resolve_config(c);
}

tcclConfig_t to_public(const Config& c) {
  tcclConfig_t p;
  std::memset(&p, 0, sizeof(p));
  p.engine = c.engine;
  p.small_max_bytes = c.small_max_bytes;
  p.vec_max_bytes = c.vec_max_bytes;
  p.stage_bytes = c.stage_bytes;
  p.stages = c.stages;
  p.store_mode = c.store_mode;
  p.consumer_warps = c.consumer_warps;
  p.ctas_per_sm = c.ctas_per_sm;
  p.wait_timeout_ms = c.wait_timeout_ms;
  p.chunk_order = c.chunk_order;
  p.stage_layout = c.stage_layout;
  p.prefetch_chunks = c.prefetch_chunks;
  p.load_policy = c.load_policy;
  p.max_chunk_bytes = c.max_chunk_bytes;
  p.ce_streams = c.ce_streams;
  p.ce_segment_bytes = c.ce_segment_bytes;
  p.ce_auto_max_cap = c.ce_auto_max_cap;
  p.reduce_order = c.reduce_order;
  p.ce_fold = c.ce_fold;
  p.ce_tail_percent = c.ce_tail_percent;
  p.reduce_slots = c.reduce_slots;
  p.ce_ar_streams = c.ce_ar_streams;
  p.ce_tail_streams = c.ce_tail_streams;
  return p;
}

bool config_ok(const tcclConfig_t& p) {
  return p.engine >= 0 && p.engine <= 5 && p.ce_streams >= 0 && p.ce_streams <= 8 &&
         p.store_mode >= 0 && p.store_mode <= 2 &&
         p.stage_bytes >= 0 && p.stages >= 0 && p.consumer_warps >= 0 && p.ctas_per_sm >= 0 &&
         p.wait_timeout_ms >= 0 && p.chunk_order >= 0 && p.chunk_order <= 3 &&
         p.prefetch_chunks >= -1 && p.load_policy >= 0 && p.load_policy <= 2 &&
         p.stage_layout >= 0 && p.stage_layout <= 2 && p.reduce_order >= 0 && p.reduce_order <= 1 &&
         p.ce_fold >= 0 && p.ce_fold <= 3 && p.ce_tail_percent >= 0 && p.ce_tail_percent <= 100 &&
         p.reduce_slots >= 0 && p.reduce_slots <= 8 && p.ce_ar_streams >= 0 && p.ce_ar_streams <= 8 &&
         p.ce_tail_streams >= 0 && p.ce_tail_streams <= 8;
}

void dump_plan(const Plan& pl, const Lowered& low) {
  std::fprintf(stderr, "[tccl] plan coll=%d P=%d count=%llu shard=%llu tasks=%zu engine=%d grid=%d "
               "threads=%d stages=%d chunk=%d smem=%zu windows=%zu\n",
               pl.coll, pl.nranks, (unsigned long long)pl.count,
               (unsigned long long)pl.shard_elems, pl.tasks.size(), low.shape.engine,
               low.shape.grid, low.shape.threads, low.shape.stages, low.shape.chunk_bytes,
               low.shape.smem, low.win.size());
  if (log_level() < 2) return;
  for (size_t i = 0; i < pl.tasks.size(); ++i) {
    const LogicalTask& t = pl.tasks[i];
    std::fprintf(stderr, "[tccl]  task %zu %s owner=%d src=%zu intervals dst=%zu intervals deps=%zu\n",
                 i, t.kind == kShardIn ? "shard-in" : "shard-out", t.exec_rank, t.src.size(),
                 t.dst.size(), t.deps.size());
  }
  for (const Window& w : low.win)
    std::fprintf(stderr, "[tccl]  win cta=%d src=%d+%llu dst=%d+%llu bytes=%u scalar=%u task=%u\n",
                 w.cta, w.src_sel, (unsigned long long)w.src_off, w.dst_sel,
                 (unsigned long long)w.dst_off, w.bytes, w.scalar, w.task);
}

}  // namespace

namespace tccl {

int log_level() {
  static int lvl = [] {
    const char* e = std::getenv("TCCL_LOG");
    return e ? std::atoi(e) : 0;
  }();
  return lvl;
}

int elem_size_of(int dtype) { return dtype == kBF16 ? 2 : 4; }

void fill_info(const Lowered& low, tcclLaunchInfo_t* info) {
  std::memset(info, 0, sizeof(*info));
  info->engine = low.shape.engine;
  info->store_mode = low.shape.store_mode;
  info->ctas = low.shape.grid;
  info->threads = low.shape.threads;
  info->stages = low.shape.stages;
  info->chunk_bytes = low.shape.chunk_bytes;
  info->windows = (int)low.win.size();
  info->tasks = low.ntasks;
  info->smem_bytes = low.shape.smem;
  const bool bulkish = low.shape.engine == kEngineBulk || low.shape.engine == kEngineTmaReduce;
  info->chunk_order = bulkish ? low.shape.order : 0;
  info->total_chunks = low.total_chunks;
  info->stage_layout = low.shape.engine == kEngineBulk ? (low.shape.rank_streamed ? 2 : 1) : 0;
}

tcclResult_t get_plan(tcclGroup* g, int coll, const void* const* send, void* const* recv,
                      size_t count, int es, int cap, CachedPlan** out, int anchor,
                      int anchor_engine) {
  PlanKey key{coll, es, (uint64_t)count, cap > 0 ? cap : 0, std::string(), anchor};
  key.anchor_engine = anchor >= 0 ? anchor_engine : 0;
  key.mod16.resize(2 * g->nranks);
  key.in_place = coll == kAllReduce;
  for (int r = 0; r < g->nranks; ++r) {
    key.mod16[r] = (char)((uintptr_t)send[r] & 15);
    key.mod16[g->nranks + r] = (char)((uintptr_t)recv[r] & 15);
    key.in_place = key.in_place && send[r] == recv[r];
  }
  auto it = g->plans.find(key);
  if (it != g->plans.end()) {
    *out = it->second.get();
    return tcclSuccess;
  }
  Plan pl = plan_collective(coll, g->nranks, count, es, 0);
  pl.in_place = key.in_place;
  pl.anchor_only = anchor >= 0;
  auto cp = std::make_unique<CachedPlan>();
  std::string why;
  std::vector<uint8_t> sm(g->nranks), rm(g->nranks);
  for (int r = 0; r < g->nranks; ++r) {
    sm[r] = (uint8_t)key.mod16[r];
    rm[r] = (uint8_t)key.mod16[g->nranks + r];
  }
  Config cfg = g->cfg;
  if (anchor >= 0) cfg.engine = anchor_engine;
  if (!lower_plan(pl, sm.data(), rm.data(), cfg, g->dev, cap, &cp->low, &why)) {
    if (log_level()) std::fprintf(stderr, "[tccl] cannot lower: %s\n", why.c_str());
    return tcclInvalidUsage;
  }
  // copy-out shard-in: the reduced chunks go to the anchor rank alone; the
  // copy engines carry them to the other ranks
  if (anchor >= 0)
    for (Window& w : cp->low.win) w.dst_sel = (int16_t)anchor;
  if (log_level()) dump_plan(pl, cp->low);
  const Lowered& low = cp->low;
  if (low.shape.engine == kEngineBulk || low.shape.engine == kEngineTmaReduce) {
    std::vector<unsigned char> host;
    size_t off_prefix = 0, off_cta = 0, off_sched = 0;
    pack_bulk_table(low, &host, &off_prefix, &off_cta, &off_sched);
    // one synchronous upload per plan: a new shape's first call must not be
    // made inside a CUDA graph capture
    if (cudaMalloc(&cp->d_table, host.size()) != cudaSuccess) return tcclCudaError;
    if (cudaMemcpy(cp->d_table, host.data(), host.size(), cudaMemcpyHostToDevice) != cudaSuccess)
      return tcclCudaError;
    cp->d_win = reinterpret_cast<const Window*>(cp->d_table);
    cp->d_prefix = reinterpret_cast<const uint64_t*>(cp->d_table + off_prefix);
    cp->d_cta_first = reinterpret_cast<const uint32_t*>(cp->d_table + off_cta);
    cp->d_sched = reinterpret_cast<unsigned long long*>(cp->d_table + off_sched);
  } else if (low.size_class == 0) {
    build_small_args<kSmallRanks, kSmallWindows>(low, g->nranks, es, &cp->small_args);
  } else {
    build_small_args<kMaxRanks, kLargeWindows>(low, g->nranks, es, &cp->small_args);
  }
  cp->anchor_only = anchor >= 0;
  *out = cp.get();
  g->plans.emplace(key, std::move(cp));
  return tcclSuccess;
}

// Launches one lowered plan on `stream` with these buffers; returns a CUDA
// error code (0 on success).
int launch_plan(tcclGroup* g, CachedPlan* cp, int coll, int dtype, int op,
                const void* const* send, void* const* recv, int es, cudaStream_t stream) {
  const Lowered& low = cp->low;
  uint32_t* mask = sm_record_slot(g);
  if (low.shape.engine == kEngineBulk || low.shape.engine == kEngineTmaReduce) {
    BulkArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int k = 0; k < g->nranks; ++k) {
      a.p.src[k] = send[k];
      a.p.dst[k] = recv[k];
    }
    a.win = cp->d_win;
    a.chunk_prefix = cp->d_prefix;
    a.cta_first = cp->d_cta_first;
    a.total_chunks = low.total_chunks;
    a.chunks_per_cta = low.chunks_per_cta;
    a.nbody = low.nbody;
    a.sched = cp->d_sched;
    a.order = low.shape.order;
    a.prefetch_chunks = low.shape.prefetch_chunks;
    a.rank_streamed = low.shape.rank_streamed;
    a.load_evict_first = low.shape.load_evict_first;
    a.arrival_order = low.shape.engine == kEngineTmaReduce && g->cfg.reduce_order == 1 ? 1 : 0;
    a.reduce_slots = low.shape.reduce_slots;
    a.anchor_only = cp->anchor_only ? 1 : 0;
    a.reduce_bufs = low.shape.reduce_bufs;
    a.status = g->d_status;
    a.sm_mask = mask;
    a.timeout_ns = (uint64_t)(g->cfg.wait_timeout_ms * 1e6);
    a.inject_timeout_ns = g->inject_ns;
    a.nranks = g->nranks;
    a.chunk_bytes = low.shape.chunk_bytes;
    a.stages = low.shape.stages;
    a.store_mode = low.shape.store_mode;
    a.consumer_warps = low.shape.consumer_warps;
    a.release_lag = low.shape.release_lag;
    a.elem_size = es;
    return low.shape.engine == kEngineBulk ? launch_bulk(coll, dtype, op, a, low.shape, stream)
                                           : launch_reduce(coll, dtype, op, a, low.shape, stream);
  }
  std::vector<unsigned char>& buf = cp->small_args;  // pointers patched in place
  if (low.size_class == 0)
    fill_small_ptrs<kSmallRanks, kSmallWindows>(&buf, g->nranks, send, recv, mask);
  else
    fill_small_ptrs<kMaxRanks, kLargeWindows>(&buf, g->nranks, send, recv, mask);
  if (coll == kAllReduce)
    return launch_small_ar(dtype, op, low.shape.engine, low.size_class, buf.data(), low.shape, stream);
  if (coll == kReduceScatter)
    return launch_small_rs(dtype, op, low.shape.engine, low.size_class, buf.data(), low.shape, stream);
  return launch_small_ag(dtype, op, low.shape.engine, low.size_class, buf.data(), low.shape, stream);
}

}  // namespace tccl

namespace {

tcclResult_t run_collective(tcclGroup* g, int coll, const void* const* send, void* const* recv,
                            size_t count, int dtype, int op, cudaStream_t stream, int cap) {
  if (!g) return tcclInvalidArgument;
  tcclResult_t v = (tcclResult_t)validate_collective_args(coll, g->nranks, send, recv, count, dtype, op);
  if (v != tcclSuccess) return v;
  if (count == 0 || is_noop(coll, g->nranks, send, recv)) {
    std::memset(&g->last, 0, sizeof(g->last));
    return tcclSuccess;
  }
  if (coll == kAllGather) op = kSum;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return tcclCudaError;
  if (cur != g->device && cudaSetDevice(g->device) != cudaSuccess) return tcclCudaError;
  const int es = elem_size_of(dtype);
  if (use_copy_out(g, coll, count, es, cap)) {
    tcclResult_t rc;
    if (coll == kAllReduce)
      rc = run_copy_out_allreduce(g, send, recv, count, dtype, op, es, stream, cap);
    else if (coll == kAllGather)
      rc = run_copy_out_allgather(g, send, recv, count, es, stream);
    else
      rc = run_copy_out_reduce_scatter(g, send, recv, count, dtype, op, es, stream, cap);
    // a reduce-scatter whose buffers the register fold cannot take runs on
    // the bulk engine below
    if (!(coll == kReduceScatter && rc == tcclInvalidUsage)) {
      if (cur != g->device) cudaSetDevice(cur);
      return rc;
    }
  }
  CachedPlan* cp = nullptr;
  tcclResult_t r = get_plan(g, coll, send, recv, count, es, cap, &cp);
  if (r == tcclSuccess && cp->low.shape.engine == kEngineTmaReduce &&
      !tma_reduce_supported(dtype, op)) {
    if (log_level())
      std::fprintf(stderr, "[tccl] the TMA-reduce engine cannot reduce dtype %d with op %d "
                           "exactly in rank order\n", dtype, op);
    r = tcclInvalidUsage;
  }
  int err = 0;
  if (r == tcclSuccess) {
    err = launch_plan(g, cp, coll, dtype, op, send, recv, es, stream);
    fill_info(cp->low, &g->last);
  }
  if (cur != g->device) cudaSetDevice(cur);
  if (r != tcclSuccess) return r;
  if (err != 0) {
    if (log_level()) std::fprintf(stderr, "[tccl] launch failed: %s\n", cudaGetErrorString((cudaError_t)err));
    return tcclCudaError;
  }
  return tcclSuccess;
}

bool to_layout(const tcclLayout_t* p, MeshLayout* l) {
  if (!p || p->ndims < 1 || p->ndims > TCCL_MAX_MESH_DIMS) return false;
  l->ndims = p->ndims;
  l->start = p->start_rank;
  for (int a = 0; a < p->ndims; ++a) {
    l->dims[a] = p->dims[a];
    l->place[a] = p->placements[a];
  }
  return true;
}

// Validates a reshard call's buffers against the plan's block sizes.
tcclResult_t check_reshard_buffers(const MeshLayout& src, const MeshLayout& dst, int nd,
                                   const uint64_t* shape, int es, const void* const* sb,
                                   void* const* dbuf) {
  if (!sb || !dbuf) return tcclInvalidArgument;
  auto block_bytes = [&](const MeshLayout& l, int m) {
    Box b = layout_box(l, nd, shape, m);
    uint64_t n = (uint64_t)es;
    for (int d = 0; d < nd; ++d) n *= b.hi[d] - b.lo[d];
    return n;
  };
  for (int m = 0; m < src.size(); ++m)
    if (!sb[m] || (uintptr_t)sb[m] % es) return tcclInvalidArgument;
  for (int m = 0; m < dst.size(); ++m)
    if (!dbuf[m] || (uintptr_t)dbuf[m] % es) return tcclInvalidArgument;
  for (int m = 0; m < dst.size(); ++m) {
    const uintptr_t a = (uintptr_t)dbuf[m];
    const uint64_t na = block_bytes(dst, m);
    for (int k = 0; k < dst.size(); ++k)
      if (k != m && ranges_overlap(a, na, (uintptr_t)dbuf[k], block_bytes(dst, k)))
        return tcclInvalidArgument;
    for (int k = 0; k < src.size(); ++k)
      if (ranges_overlap(a, na, (uintptr_t)sb[k], block_bytes(src, k))) return tcclInvalidArgument;
  }
  return tcclSuccess;
}

}  // namespace

extern "C" {

const char* tcclGetErrorString(tcclResult_t r) {
  switch (r) {
    case tcclSuccess: return "success";
    case tcclInvalidArgument: return "invalid argument";
    case tcclInvalidUsage: return "invalid usage";
    case tcclCudaError: return "CUDA error";
    case tcclDeviceTimeout: return "device-side wait timed out";
    case tcclInternalError: return "internal error";
  }
  return "unknown result code";
}

tcclResult_t tcclGetVersion(int* version) {
  if (!version) return tcclInvalidArgument;
  *version = TCCL_VERSION;
  return tcclSuccess;
}

tcclResult_t tcclGroupCreate(int nranks, tcclGroup_t* out) {
  if (!out || nranks < 1 || nranks > TCCL_MAX_RANKS) return tcclInvalidArgument;
  *out = nullptr;
  auto g = std::make_unique<tcclGroup>();
  g->nranks = nranks;
  if (cudaGetDevice(&g->device) != cudaSuccess) return tcclCudaError;
  if (cudaDeviceGetAttribute(&g->dev.sm_count, cudaDevAttrMultiProcessorCount, g->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&g->dev.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, g->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&g->dev.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, g->device) != cudaSuccess)
    return tcclCudaError;
  g->cfg = config_from_env();
  if (const char* e = std::getenv("TCCL_RMSNORM_CLUSTER")) g->rms_cluster_enabled = std::atoi(e) != 0;
  if (prepare_bulk_kernels((size_t)g->dev.smem_optin) != 0) return tcclCudaError;
  if (prepare_reshard_kernels((size_t)g->dev.smem_optin) != 0) return tcclCudaError;
  if (cudaMalloc(&g->d_status, 64) != cudaSuccess) return tcclCudaError;
  const size_t sm_bytes = sizeof(uint32_t) * kSmSlots * kSmSlotWords;
  if (cudaMalloc(&g->d_sm_mask, sm_bytes) != cudaSuccess) {
    cudaFree(g->d_status);
    return tcclCudaError;
  }
  if (cudaMemset(g->d_status, 0, 64) != cudaSuccess || cudaMemset(g->d_sm_mask, 0, sm_bytes) != cudaSuccess) {
    cudaFree(g->d_status);
    cudaFree(g->d_sm_mask);
    return tcclCudaError;
  }
  std::memset(&g->last, 0, sizeof(g->last));
  *out = g.release();
  return tcclSuccess;
}

tcclResult_t tcclGroupDestroy(tcclGroup_t g) {
  if (!g) return tcclInvalidArgument;
  cudaDeviceSynchronize();
  g->plans.clear();
  g->reshards.clear();
  for (cudaStream_t st : g->ce_streams) cudaStreamDestroy(st);
  for (cudaEvent_t e : g->ce_seg_events) cudaEventDestroy(e);
  for (cudaEvent_t e : g->ce_done_events) cudaEventDestroy(e);
  if (g->ce_fork_event) cudaEventDestroy(g->ce_fork_event);
  cudaFree(g->d_status);
  cudaFree(g->d_sm_mask);
  delete g;
  return tcclSuccess;
}

tcclResult_t tcclGroupGetConfig(tcclGroup_t g, tcclConfig_t* cfg) {
  if (!g || !cfg) return tcclInvalidArgument;
  *cfg = to_public(g->cfg);
  return tcclSuccess;
}

tcclResult_t tcclGroupSetConfig(tcclGroup_t g, const tcclConfig_t* cfg) {
  if (!g || !cfg || !config_ok(*cfg)) return tcclInvalidArgument;
  cudaDeviceSynchronize();  // plans in flight keep their device tables until done
  g->cfg = from_public(*cfg);
  g->plans.clear();
  g->reshards.clear();
  return tcclSuccess;
}

tcclResult_t tcclAllReduce(tcclGroup_t g, const void* const sendbufs[], void* const recvbufs[],
                           size_t count, tcclDataType_t datatype, tcclRedOp_t op,
                           cudaStream_t stream, int cta_cap) {
  return run_collective(g, kAllReduce, sendbufs, recvbufs, count, datatype, op, stream, cta_cap);
}

tcclResult_t tcclReduceScatter(tcclGroup_t g, const void* const sendbufs[],
                               void* const recvbufs[], size_t recvcount,
                               tcclDataType_t datatype, tcclRedOp_t op, cudaStream_t stream,
                               int cta_cap) {
  return run_collective(g, kReduceScatter, sendbufs, recvbufs, recvcount, datatype, op, stream,
                        cta_cap);
}

tcclResult_t tcclAllGather(tcclGroup_t g, const void* const sendbufs[], void* const recvbufs[],
                           size_t sendcount, tcclDataType_t datatype, cudaStream_t stream,
                           int cta_cap) {
  return run_collective(g, kAllGather, sendbufs, recvbufs, sendcount, datatype, kSum, stream,
                        cta_cap);
}

tcclResult_t tcclGroupQueryError(tcclGroup_t g, tcclResult_t* async_status) {
  if (!g || !async_status) return tcclInvalidArgument;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return tcclCudaError;
  if (cur != g->device) cudaSetDevice(g->device);
  int st = 0;
  bool ok = cudaDeviceSynchronize() == cudaSuccess &&
            cudaMemcpy(&st, g->d_status, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess &&
            cudaMemset(g->d_status, 0, sizeof(int)) == cudaSuccess;
  if (cur != g->device) cudaSetDevice(cur);
  if (!ok) return tcclCudaError;
  *async_status = (tcclResult_t)st;
  return tcclSuccess;
}

tcclResult_t tcclGetLastLaunchInfo(tcclGroup_t g, tcclLaunchInfo_t* info) {
  if (!g || !info) return tcclInvalidArgument;
  *info = g->last;
  return tcclSuccess;
}

tcclResult_t tcclGroupRecordSms(tcclGroup_t g, int enable) {
  if (!g) return tcclInvalidArgument;
  g->record_sms = enable != 0;
  return tcclSuccess;
}

}  // extern "C"

namespace {

// Reads and clears the SM record: the distinct SMs of each recorded launch
// (up to max_launches of them) and of all launches together.
tcclResult_t read_sm_record(tcclGroup_t g, int* per_launch, int max_launches, int* n_launches,
                            int* distinct_sms) {
  std::vector<uint32_t> m((size_t)kSmSlots * kSmSlotWords);
  const size_t bytes = m.size() * sizeof(uint32_t);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(m.data(), g->d_sm_mask, bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(g->d_sm_mask, 0, bytes) != cudaSuccess)
    return tcclCudaError;
  const int launches = g->sm_launches;
  g->sm_launches = 0;
  uint32_t all[kSmSlotWords] = {0};
  for (int s = 0; s < kSmSlots; ++s) {
    int n = 0;
    for (int w = 0; w < kSmSlotWords; ++w) {
      const uint32_t v = m[(size_t)s * kSmSlotWords + w];
      all[w] |= v;
      n += __builtin_popcount(v);
    }
    if (per_launch && s < max_launches && s < launches) per_launch[s] = n;
  }
  int n = 0;
  for (uint32_t w : all) n += __builtin_popcount(w);
  if (distinct_sms) *distinct_sms = n;
  if (n_launches) *n_launches = launches;
  return tcclSuccess;
}

}  // namespace

extern "C" {

tcclResult_t tcclGroupReadSmRecord(tcclGroup_t g, int* distinct_sms) {
  if (!g || !distinct_sms) return tcclInvalidArgument;
  return read_sm_record(g, nullptr, 0, nullptr, distinct_sms);
}

tcclResult_t tcclGroupReadSmRecordLaunches(tcclGroup_t g, int* per_launch, int max_launches,
                                           int* n_launches, int* distinct_sms) {
  if (!g || !n_launches || !distinct_sms || max_launches < 0 || (max_launches > 0 && !per_launch))
    return tcclInvalidArgument;
  return read_sm_record(g, per_launch, max_launches, n_launches, distinct_sms);
}

tcclResult_t tcclReshard(tcclGroup_t g, const void* const srcbufs[], const tcclLayout_t* src,
                         void* const dstbufs[], const tcclLayout_t* dst, int tensor_ndims,
                         const size_t* tensor_shape, tcclDataType_t datatype,
                         cudaStream_t stream, int cta_cap) {
  if (!g || !tensor_shape || tensor_ndims < 1 || tensor_ndims > TCCL_MAX_TENSOR_DIMS)
    return tcclInvalidArgument;
  if (datatype < tcclFloat32 || datatype > tcclInt32) return tcclInvalidArgument;
  MeshLayout sl, dl;
  if (!to_layout(src, &sl) || !to_layout(dst, &dl)) return tcclInvalidArgument;
  uint64_t shape[TCCL_MAX_TENSOR_DIMS];
  for (int d = 0; d < tensor_ndims; ++d) shape[d] = tensor_shape[d];
  std::string why;
  if (!check_layout(sl, tensor_ndims, shape, &why) || !check_layout(dl, tensor_ndims, shape, &why) ||
      sl.start + sl.size() > g->nranks || dl.start + dl.size() > g->nranks) {
    if (log_level()) std::fprintf(stderr, "[tccl] reshard: %s\n", why.empty() ? "mesh outside the group" : why.c_str());
    return tcclInvalidArgument;
  }
  const int es = elem_size_of(datatype);
  tcclResult_t v = check_reshard_buffers(sl, dl, tensor_ndims, shape, es, srcbufs, dstbufs);
  if (v != tcclSuccess) return v;
  // plan cache key: layouts, shape, element size, cap, buffer alignments
  std::string key;
  auto put = [&](const void* p, size_t n) { key.append(static_cast<const char*>(p), n); };
  put(&sl, sizeof(sl));
  put(&dl, sizeof(dl));
  put(&tensor_ndims, sizeof(int));
  put(shape, sizeof(uint64_t) * tensor_ndims);
  put(&es, sizeof(int));
  put(&cta_cap, sizeof(int));
  // the group's engine setting picks between the bulk ring and warp copies
  put(&g->cfg.engine, sizeof(int));
  std::vector<uint8_t> sm(sl.size()), dm(dl.size());
  for (int m = 0; m < sl.size(); ++m) sm[m] = (uint8_t)((uintptr_t)srcbufs[m] & 15);
  for (int m = 0; m < dl.size(); ++m) dm[m] = (uint8_t)((uintptr_t)dstbufs[m] & 15);
  put(sm.data(), sm.size());
  put(dm.data(), dm.size());
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return tcclCudaError;
  if (cur != g->device && cudaSetDevice(g->device) != cudaSuccess) return tcclCudaError;
  tcclResult_t result = tcclSuccess;
  auto it = g->reshards.find(key);
  CachedReshard* cr = nullptr;
  if (it != g->reshards.end()) {
    cr = it->second.get();
  } else {
    auto fresh = std::make_unique<CachedReshard>();
    if (!plan_reshard(sl, dl, tensor_ndims, shape, es, sm.data(), dm.data(), g->dev.sm_count,
                      cta_cap, g->cfg.engine, (size_t)g->dev.smem_optin, &fresh->plan, &why)) {
      if (log_level()) std::fprintf(stderr, "[tccl] reshard: %s\n", why.c_str());
      result = tcclInvalidArgument;
    } else {
      // device table: windows, unit prefix, then two zeroed claim words
      const size_t wb = fresh->plan.win.size() * sizeof(ReshardWindow);
      const size_t pb = fresh->plan.unit_prefix.size() * sizeof(uint64_t);
      std::vector<unsigned char> host(wb + pb + 16, 0);
      if (wb) std::memcpy(host.data(), fresh->plan.win.data(), wb);
      std::memcpy(host.data() + wb, fresh->plan.unit_prefix.data(), pb);
      if (cudaMalloc(&fresh->d_table, host.size()) != cudaSuccess ||
          cudaMemcpy(fresh->d_table, host.data(), host.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        result = tcclCudaError;
      else {
        cr = fresh.get();
        g->reshards.emplace(key, std::move(fresh));
      }
    }
  }
  if (result == tcclSuccess && !cr->plan.win.empty()) {
    ReshardArgs a;
    std::memset(&a, 0, sizeof(a));
    const size_t wb = cr->plan.win.size() * sizeof(ReshardWindow);
    const size_t pb = cr->plan.unit_prefix.size() * sizeof(uint64_t);
    a.win = reinterpret_cast<const ReshardWindow*>(cr->d_table);
    a.unit_prefix = reinterpret_cast<const uint64_t*>(cr->d_table + wb);
    a.sched = reinterpret_cast<unsigned long long*>(cr->d_table + wb + pb);
    for (int m = 0; m < sl.size(); ++m) a.src[m] = srcbufs[m];
    for (int m = 0; m < dl.size(); ++m) a.dst[m] = dstbufs[m];
    a.sm_mask = sm_record_slot(g);
    a.status = g->d_status;
    a.timeout_ns = (uint64_t)(g->cfg.wait_timeout_ms * 1e6);
    a.inject_timeout_ns = g->inject_ns;
    a.nwin = (int)cr->plan.win.size();
    a.elem_size = es;
    const int rc = cr->plan.engine == kReshardBulk
                       ? launch_reshard_bulk(a, cr->plan.grid, cr->plan.smem, cta_cap <= 0, stream)
                       : launch_reshard(a, cr->plan.grid, cta_cap <= 0, stream);
    if (rc != 0) result = tcclCudaError;
    std::memset(&g->last, 0, sizeof(g->last));
    const bool bulk = cr->plan.engine == kReshardBulk;
    g->last.engine = bulk ? kEngineBulk : kEngineWarp;
    g->last.ctas = cr->plan.grid;
    g->last.threads = cr->plan.threads;
    g->last.stages = bulk ? kReshardBulkStages : 0;
    g->last.chunk_bytes = bulk ? kReshardBulkSegBytes : kReshardSegBytes;
    g->last.smem_bytes = cr->plan.smem;
    g->last.total_chunks = cr->plan.unit_prefix.back();
    g->last.windows = (int)cr->plan.win.size();
    g->last.tasks = (int)cr->plan.transfers.size();
  }
  if (cur != g->device) cudaSetDevice(cur);
  return result;
}

tcclResult_t tcclAllReduceRMSNorm(tcclGroup_t g, const void* const sendbufs[],
                                  void* const recvbufs[], size_t rows, size_t hidden,
                                  const void* gamma, float eps, tcclDataType_t datatype,
                                  cudaStream_t stream, int cta_cap) {
  if (!g) return tcclInvalidArgument;
  if (datatype != tcclFloat32 && datatype != tcclBfloat16) return tcclInvalidArgument;
  const int es = elem_size_of(datatype);
  const size_t vec_elems = 16 / es;
  const size_t max_hidden = std::min<size_t>((size_t)kRmsMaxThreads * kRmsMaxVectors * vec_elems,
                                             (size_t)16384);
  if (hidden == 0 || hidden % vec_elems || hidden > max_hidden || !(eps >= 0.f)) return tcclInvalidArgument;
  if (rows > (SIZE_MAX / 4) / hidden) return tcclInvalidArgument;
  tcclResult_t v = (tcclResult_t)validate_collective_args(kAllReduce, g->nranks, sendbufs, recvbufs,
                                                          rows * hidden, datatype, kSum);
  if (v != tcclSuccess) return v;
  if (rows == 0) return tcclSuccess;
  if (!gamma || (uintptr_t)gamma % 16) return tcclInvalidArgument;
  for (int r = 0; r < g->nranks; ++r) {
    if ((uintptr_t)sendbufs[r] % 16 || (uintptr_t)recvbufs[r] % 16) return tcclInvalidArgument;
    if (ranges_overlap((uintptr_t)gamma, hidden * es, (uintptr_t)recvbufs[r], rows * hidden * es))
      return tcclInvalidArgument;
  }
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return tcclCudaError;
  if (cur != g->device && cudaSetDevice(g->device) != cudaSuccess) return tcclCudaError;
  RmsArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < g->nranks; ++r) {
    a.p.src[r] = sendbufs[r];
    a.p.dst[r] = recvbufs[r];
  }
  a.gamma = gamma;
  a.sm_mask = sm_record_slot(g);
  a.rows = rows;
  a.hidden = (uint32_t)hidden;
  a.eps = eps;
  a.nranks = g->nranks;
  const size_t nvec = hidden / vec_elems;
  // Few rows: a cluster of C CTAs shares each row, so a decode-sized call
  // uses more than one SM per row. C is the largest of 8, 4, 2 whose grid
  // (rows x C CTAs, two resident per SM) fits in one wave; each CTA's slice
  // must fit its 4 vectors per thread.
  int C = kRmsCluster;
  while (C > 2 && (rows * (size_t)C > (size_t)g->dev.sm_count * 2 || (cta_cap > 0 && cta_cap < C)))
    C /= 2;
  const bool cluster = g->rms_cluster_enabled && rows * (size_t)C <= (size_t)g->dev.sm_count * 2 &&
                       (cta_cap <= 0 || cta_cap >= C) &&
                       (nvec + C - 1) / C <= (size_t)4 * kRmsClusterThreads;
  int err;
  std::memset(&g->last, 0, sizeof(g->last));
  if (cluster) {
    uint64_t clusters = std::min<uint64_t>(rows, (uint64_t)g->dev.sm_count * 8 / C);
    if (cta_cap > 0) clusters = std::min<uint64_t>(clusters, (uint64_t)(cta_cap / C));
    err = launch_rmsnorm_cluster(datatype, a, (int)clusters, C, cta_cap <= 0, stream);
    g->last.ctas = (int)(clusters * C);
    g->last.threads = kRmsClusterThreads;
  } else {
    const int vectors = nvec > (size_t)4 * kRmsMaxThreads ? 8 : 4;
    int threads = (int)std::min<size_t>(kRmsMaxThreads, ((nvec + vectors - 1) / vectors + 31) / 32 * 32);
    threads = std::max(threads, 32);
    // up to 8 rows per SM: one CTA per row; up to 16: 8 CTAs per SM taking
    // every gridDim-th row (the block scheduler spreads the CTAs). More rows
    // than that, or than a cap allows: a grid of the CTAs that fit on the SMs
    // at once, which claim rows from a counter in the group's status block
    // (bytes 32..47), so the SMs finish together
    uint64_t grid = std::min<uint64_t>(rows, (uint64_t)g->dev.sm_count * 8);
    if (cta_cap > 0) grid = std::min<uint64_t>(grid, (uint64_t)cta_cap);
    if (rows > grid && (cta_cap > 0 || rows > (uint64_t)g->dev.sm_count * 16)) {
      const int per_sm = rmsnorm_ctas_per_sm(datatype, threads, vectors, hidden * es);
      if (per_sm > 0) grid = std::min<uint64_t>(grid, (uint64_t)g->dev.sm_count * per_sm);
      a.claim = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(g->d_status) + 32);
    }
    err = launch_rmsnorm(datatype, a, (int)grid, threads, vectors, cta_cap <= 0, stream);
    g->last.ctas = (int)grid;
    g->last.threads = threads;
  }
  if (cur != g->device) cudaSetDevice(cur);
  return err == 0 ? tcclSuccess : tcclCudaError;
}

tcclResult_t tcclReshardInspect(const tcclLayout_t* src, const tcclLayout_t* dst,
                                int tensor_ndims, const size_t* tensor_shape,
                                tcclDataType_t datatype, const void* const srcbufs[],
                                void* const dstbufs[], int sm_count, int cta_cap,
                                int64_t* transfers, int max_transfers, int* n_transfers,
                                int64_t* bytes_read, int64_t* bytes_written, int* n_windows) {
  if (!tensor_shape || tensor_ndims < 1 || tensor_ndims > TCCL_MAX_TENSOR_DIMS || !n_transfers ||
      !bytes_read || !bytes_written || !n_windows || sm_count < 1)
    return tcclInvalidArgument;
  if (datatype < tcclFloat32 || datatype > tcclInt32) return tcclInvalidArgument;
  MeshLayout sl, dl;
  if (!to_layout(src, &sl) || !to_layout(dst, &dl)) return tcclInvalidArgument;
  uint64_t shape[TCCL_MAX_TENSOR_DIMS];
  for (int d = 0; d < tensor_ndims; ++d) shape[d] = tensor_shape[d];
  std::string why;
  if (!check_layout(sl, tensor_ndims, shape, &why) || !check_layout(dl, tensor_ndims, shape, &why))
    return tcclInvalidArgument;
  const int es = elem_size_of(datatype);
  tcclResult_t v = check_reshard_buffers(sl, dl, tensor_ndims, shape, es, srcbufs, dstbufs);
  if (v != tcclSuccess) return v;
  std::vector<uint8_t> sm(sl.size()), dm(dl.size());
  for (int m = 0; m < sl.size(); ++m) sm[m] = (uint8_t)((uintptr_t)srcbufs[m] & 15);
  for (int m = 0; m < dl.size(); ++m) dm[m] = (uint8_t)((uintptr_t)dstbufs[m] & 15);
  ReshardPlan plan;
  if (!plan_reshard(sl, dl, tensor_ndims, shape, es, sm.data(), dm.data(), sm_count, cta_cap,
                    kEngineAuto, 232448, &plan, &why))
    return tcclInvalidArgument;
  *n_transfers = (int)plan.transfers.size();
  *bytes_read = (int64_t)plan.bytes_read;
  *bytes_written = (int64_t)plan.bytes_written;
  *n_windows = (int)plan.win.size();
  if (transfers) {
    for (int i = 0; i < std::min(max_transfers, (int)plan.transfers.size()); ++i) {
      const ReshardTransfer& t = plan.transfers[i];
      int64_t* o = transfers + 10 * (size_t)i;
      o[0] = t.src_rank;
      o[1] = (int64_t)t.dst_mask;
      for (int d = 0; d < 4; ++d) {
        o[2 + d] = d < tensor_ndims ? (int64_t)t.box.lo[d] : 0;
        o[6 + d] = d < tensor_ndims ? (int64_t)t.box.hi[d] : 0;
      }
    }
  }
  return tcclSuccess;
}

tcclResult_t tcclGroupInjectWaitTimeout(tcclGroup_t g, int enable, double timeout_ms) {
  if (!g || (enable && timeout_ms <= 0)) return tcclInvalidArgument;
  g->inject_ns = enable ? (uint64_t)(timeout_ms * 1e6) : 0;
  return tcclSuccess;
}

tcclResult_t tcclCopyOutInspect(int coll, int nranks, const void* const sendbufs[],
                                void* const recvbufs[], size_t count, tcclDataType_t datatype,
                                int cta_cap, int sm_count, const tcclConfig_t* cfg, int* copy_out,
                                int* register_fold, int* segments, size_t* segment_elems,
                                int* wide_folds) {
  if (!copy_out || !register_fold || !segments || !segment_elems || !wide_folds || sm_count < 1)
    return tcclInvalidArgument;
  if (cfg && !config_ok(*cfg)) return tcclInvalidArgument;
  tcclResult_t v = (tcclResult_t)validate_collective_args(coll, nranks, sendbufs, recvbufs, count, datatype, 0);
  if (v != tcclSuccess) return v;
  *copy_out = *register_fold = *segments = *wide_folds = 0;
  *segment_elems = 0;
  if (count == 0 || is_noop(coll, nranks, sendbufs, recvbufs)) return tcclSuccess;
  const int es = elem_size_of(datatype);
  const Config c = cfg ? from_public(*cfg) : resolve_config(Config());
  if (!copy_out_chosen(c, sm_count, nranks, coll, count, es, cta_cap)) return tcclSuccess;
  *copy_out = 1;
  const std::vector<uint8_t> sm = mod16_of(nranks, sendbufs);
  const std::vector<uint8_t> rm = mod16_of(nranks, (const void* const*)recvbufs);
  if (coll == kAllReduce) {
    size_t seg = 0;
    int nseg = 0;
    copy_out_segments(c, count, es, &seg, &nseg);
    *segments = nseg;
    *segment_elems = seg;
    *register_fold = allreduce_register_fold(c, nranks, sm.data(), rm.data(), count, es, seg) ? 1 : 0;
    // the fold's arguments segment by segment, as the call would make them
    for (int k = 0; k < nseg && *register_fold; ++k) {
      AnchorArgs a;
      allreduce_segment_args(&a, nranks, sendbufs, recvbufs[0], (size_t)k * seg,
                             k == nseg - 1 ? count - (size_t)k * seg : seg, es);
      *wide_folds += a.wide;
    }
  } else if (coll == kReduceScatter) {
    *register_fold = register_fold_ok(coll, nranks, sm.data(), rm.data(), count, es, 0) ? 1 : 0;
    *copy_out = *register_fold;  // otherwise the bulk engine runs it
    *segments = *register_fold;
    *segment_elems = *register_fold ? count : 0;
    if (*register_fold) {
      AnchorArgs a;
      reduce_scatter_args(&a, nranks, sendbufs, recvbufs, count, es);
      *wide_folds = a.wide;
    }
  }
  return tcclSuccess;
}

tcclResult_t tcclPlanInspect(int coll, int nranks, const void* const sendbufs[],
                             void* const recvbufs[], size_t count, tcclDataType_t datatype,
                             int cta_cap, int sm_count, int smem_per_block,
                             const tcclConfig_t* cfg, int64_t* windows, int max_windows,
                             int* n_windows, int* n_tasks, tcclLaunchInfo_t* info) {
  if (!n_windows || !n_tasks || !info || sm_count < 1 || smem_per_block < 1) return tcclInvalidArgument;
  if (cfg && !config_ok(*cfg)) return tcclInvalidArgument;
  tcclResult_t v = (tcclResult_t)validate_collective_args(coll, nranks, sendbufs, recvbufs, count, datatype, 0);
  if (v != tcclSuccess) return v;
  *n_windows = 0;
  *n_tasks = 0;
  std::memset(info, 0, sizeof(*info));
  if (count == 0) return tcclSuccess;
  const int es = elem_size_of(datatype);
  Plan pl = plan_collective(coll, nranks, count, es, 0);
  std::vector<uint8_t> sm(nranks), rm(nranks);
  pl.in_place = coll == kAllReduce;
  for (int r = 0; r < nranks; ++r) {
    sm[r] = (uint8_t)((uintptr_t)sendbufs[r] & 15);
    rm[r] = (uint8_t)((uintptr_t)recvbufs[r] & 15);
    pl.in_place = pl.in_place && sendbufs[r] == recvbufs[r];
  }
  DeviceDesc dev;
  dev.sm_count = sm_count;
  dev.smem_optin = smem_per_block;
  dev.smem_per_sm = smem_per_block + 1024;
  Config c = cfg ? from_public(*cfg) : resolve_config(Config());
  Lowered low;
  std::string why;
  if (!lower_plan(pl, sm.data(), rm.data(), c, dev, cta_cap, &low, &why)) return tcclInvalidUsage;
  *n_tasks = (int)pl.tasks.size();
  *n_windows = (int)low.win.size();
  fill_info(low, info);
  if (windows) {
    for (int i = 0; i < std::min(max_windows, (int)low.win.size()); ++i) {
      const Window& w = low.win[i];
      int64_t* o = windows + 8 * (size_t)i;
      o[0] = w.cta;
      o[1] = w.src_sel;
      o[2] = (int64_t)w.src_off;
      o[3] = w.dst_sel;
      o[4] = (int64_t)w.dst_off;
      o[5] = w.bytes;
      o[6] = w.scalar;
      o[7] = w.task;
    }
  }
  return tcclSuccess;
}

}  // extern "C"
