// Host side of the copy-out engine: Auto's choice, the segment pipeline of
// the allreduce (register-load fold or TMA shard-in into one anchor rank,
// then device-to-device copies on the group's copy streams), the
// reduce-scatter on the register fold, and the all-gather as copies only.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "copy_out.h"
#include "group.h"
#include "internal.h"
#include "plan.h"

namespace tccl {

bool use_copy_out(const tcclGroup* g, int coll, size_t count, int es, int cap) {
  return copy_out_chosen(g->cfg, g->dev.sm_count, g->nranks, coll, count, es, cap);
}

std::vector<uint8_t> mod16_of(int n, const void* const* p) {
  std::vector<uint8_t> m(n);
  for (int k = 0; k < n; ++k) m[k] = (uint8_t)((uintptr_t)p[k] & 15);
  return m;
}

namespace {

// bf16 sums in the register-load fold: the mixed-precision add unless
// TCCL_BF16_FOLD=packed asks for the packed fp32 adds (the same bits).
int mixed_bf16_fold() {
  static const int v = [] {
    const char* e = std::getenv("TCCL_BF16_FOLD");
    return (e && std::string(e) == "packed") ? 0 : 1;
  }();
  return v;
}

// The group's copy streams, the per-segment events and the join events,
// created on first use (so a group that never uses the engine holds none).
tcclResult_t ensure_ce_resources(tcclGroup* g, int segments) {
  const int ns = g->cfg.ce_streams;
  while ((int)g->ce_streams.size() < ns) {
    cudaStream_t st;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return tcclCudaError;
    g->ce_streams.push_back(st);
  }
  while ((int)g->ce_done_events.size() < ns) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return tcclCudaError;
    g->ce_done_events.push_back(e);
  }
  while ((int)g->ce_seg_events.size() < segments) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return tcclCudaError;
    g->ce_seg_events.push_back(e);
  }
  if (!g->ce_fork_event &&
      cudaEventCreateWithFlags(&g->ce_fork_event, cudaEventDisableTiming) != cudaSuccess)
    return tcclCudaError;
  return tcclSuccess;
}

// Makes `stream` wait for everything queued on the first `used` copy streams.
int join_ce_streams(tcclGroup* g, int used, cudaStream_t stream) {
  int err = 0;
  for (int j = 0; j < used; ++j) {
    int e = cudaEventRecord(g->ce_done_events[j], g->ce_streams[j]);
    if (!e) e = cudaStreamWaitEvent(stream, g->ce_done_events[j], 0);
    if (e && !err) err = e;
  }
  return err;
}

}  // namespace

// The register fold's arguments for one allreduce segment or one
// reduce-scatter (both declared in copy_out.h).
void allreduce_segment_args(AnchorArgs* a, int nranks, const void* const* send,
                            void* anchor_recv, size_t off, size_t n, int es) {
  std::memset(a, 0, sizeof(*a));
  a->nranks = nranks;
  a->njobs = 1;
  const uintptr_t mod = (uintptr_t)anchor_recv & 15;
  const size_t bytes = n * es;
  a->head_bytes = std::min(bytes, (size_t)((16 - mod) & 15));
  a->nvec = (bytes - a->head_bytes) / 16;
  a->tail_bytes = bytes - a->head_bytes - a->nvec * 16;
  for (int k = 0; k < nranks; ++k) a->p.src[k] = static_cast<const char*>(send[k]) + off * es;
  a->p.dst[0] = static_cast<char*>(anchor_recv) + off * es;
  a->wide = anchor_wide_ok(*a) ? 1 : 0;
}

void reduce_scatter_args(AnchorArgs* a, int nranks, const void* const* send,
                         void* const* recv, size_t rc, int es) {
  std::memset(a, 0, sizeof(*a));
  a->nranks = nranks;
  a->njobs = nranks;
  const uintptr_t mod = (uintptr_t)recv[0] & 15;
  const size_t bytes = rc * (size_t)es;
  a->job_src_stride = bytes;
  a->head_bytes = std::min(bytes, (size_t)((16 - mod) & 15));
  a->nvec = (bytes - a->head_bytes) / 16;
  a->tail_bytes = bytes - a->head_bytes - a->nvec * 16;
  for (int k = 0; k < nranks; ++k) {
    a->p.src[k] = send[k];
    a->p.dst[k] = recv[k];
  }
  a->wide = anchor_wide_ok(*a) ? 1 : 0;
}

// Allreduce on the copy-out engine. The message is cut into segments
// (copy_out_segments: at most ce_segment_bytes per rank, at least four of at
// least 4 MiB where the message allows, offsets multiples of 256 bytes, so
// every segment has the same alignment). Each segment's shard-in kernel folds the P
// ranks in ascending order into the anchor rank's (rank 0's) receive buffer
// alone; an event after it releases the device-to-device copies of that
// segment from the anchor to ranks 1..P-1 on the group's copy streams, so the
// copy engines fan segment s out while the SMs reduce segment s+1. In place
// is safe: segment s of a rank is overwritten only after the kernel that read
// it has finished.
//
// The shard-in kernel is the register-load anchor fold when every send buffer
// and the anchor's receive buffer share their address mod 16, else the bulk
// engine's TMA pipeline with every window pointed at the anchor.
tcclResult_t run_copy_out_allreduce(tcclGroup* g, const void* const* send, void* const* recv,
                                    size_t count, int dtype, int op, int es, cudaStream_t stream,
                                    int cap) {
  const int P = g->nranks;
  const int anchor = 0;
  size_t seg = 0;
  int nseg = 0;
  copy_out_segments(g->cfg, count, es, &seg, &nseg);
  tcclResult_t r = ensure_ce_resources(g, nseg);
  if (r != tcclSuccess) return r;
  std::vector<const void*> s_ptr(P);
  std::vector<void*> r_ptr(P);
  auto at = [&](size_t off) {
    for (int k = 0; k < P; ++k) {
      s_ptr[k] = static_cast<const char*>(send[k]) + off * es;
      r_ptr[k] = static_cast<char*>(recv[k]) + off * es;
    }
  };
  // ce_fold = 3: bulk reductions into the anchor, for the pairs the copy
  // hardware reduces exactly; any other pair folds as under Auto
  const bool tma_reduce = g->cfg.ce_fold == kFoldTmaReduce && tma_reduce_supported(dtype, op);
  Config fold_cfg = g->cfg;
  if (fold_cfg.ce_fold == kFoldTmaReduce && !tma_reduce) fold_cfg.ce_fold = kFoldAuto;
  const bool fast = !tma_reduce &&
                    allreduce_register_fold(fold_cfg, P, mod16_of(P, send).data(),
                                            mod16_of(P, (const void* const*)recv).data(), count,
                                            es, seg);
  const int anchor_engine = tma_reduce ? kEngineTmaReduce : kEngineBulk;
  const size_t tail_n = count - (size_t)(nseg - 1) * seg;
  // TMA fallback: both plans (full segments, ragged tail) before any launch,
  // since a new plan's table upload is synchronous
  CachedPlan* full = nullptr;
  CachedPlan* tail = nullptr;
  if (!fast) {
    at(0);
    r = get_plan(g, kAllReduce, s_ptr.data(), r_ptr.data(), nseg > 1 ? seg : tail_n, es, cap, &full, anchor,
                 anchor_engine);
    if (r == tcclSuccess && nseg > 1 && tail_n != seg) {
      at((size_t)(nseg - 1) * seg);
      r = get_plan(g, kAllReduce, s_ptr.data(), r_ptr.data(), tail_n, es, cap, &tail, anchor,
                   anchor_engine);
    }
    if (r != tcclSuccess) return r;
  }
  const int U = anchor_vectors_per_thread(P);
  int fast_grid = 0;
  AnchorArgs aa;
  // the copies of every segment but the last run beside the next segment's
  // fold, the last segment's beside nothing: each has its own stream count
  int mid_streams = 0, tail_streams = 0;
  copy_out_streams(g->cfg, P, cap, &mid_streams, &tail_streams);
  const int used = P > 1 ? std::max(mid_streams, tail_streams) : 0;
  int err = 0, copies = 0, wide_folds = 0;
  for (int sgi = 0; sgi < nseg && !err; ++sgi) {
    const size_t off = (size_t)sgi * seg;
    const size_t n = sgi == nseg - 1 ? tail_n : seg;
    at(off);
    if (fast) {
      allreduce_segment_args(&aa, P, send, recv[anchor], off, n, es);
      aa.mixed_bf16 = mixed_bf16_fold();
      wide_folds += aa.wide;
      const uint64_t per_cta = (uint64_t)kAnchorThreads * (aa.wide ? anchor_vectors_per_thread(P, true, dtype) : U);
      uint64_t grid = std::max<uint64_t>(1, (aa.nvec + per_cta - 1) / per_cta);
      grid = std::min<uint64_t>(grid, cap > 0 ? (uint64_t)cap : (uint64_t)g->dev.sm_count);
      fast_grid = std::max(fast_grid, (int)grid);
      aa.sm_mask = sm_record_slot(g);
      err = launch_anchor_reduce(dtype, op, aa, (int)grid, cap <= 0, stream);
    } else {
      CachedPlan* cp = (sgi == nseg - 1 && tail) ? tail : full;
      err = launch_plan(g, cp, kAllReduce, dtype, op, s_ptr.data(), r_ptr.data(), es, stream);
    }
    if (err || used == 0) continue;
    const int seg_streams = sgi == nseg - 1 ? tail_streams : mid_streams;
    err = cudaEventRecord(g->ce_seg_events[sgi], stream);
    for (int j = 0; j < seg_streams && !err; ++j) err = cudaStreamWaitEvent(g->ce_streams[j], g->ce_seg_events[sgi], 0);
    int j = 0;
    for (int k = 0; k < P && !err; ++k) {
      if (k == anchor) continue;
      err = cudaMemcpyAsync(r_ptr[k], r_ptr[anchor], n * es, cudaMemcpyDeviceToDevice, g->ce_streams[j]);
      j = (j + 1) % seg_streams;
      ++copies;
    }
  }
  const int jerr = used ? join_ce_streams(g, used, stream) : 0;
  if (!err) err = jerr;
  if (fast) {
    std::memset(&g->last, 0, sizeof(g->last));
    g->last.store_mode = kStoreVec;
    g->last.ctas = fast_grid;
    g->last.threads = kAnchorThreads;
  } else {
    fill_info(full->low, &g->last);
  }
  g->last.engine = kEngineCopyOut;
  g->last.ce_segments = nseg;
  g->last.ce_copies = copies;
  g->last.ce_wide_folds = wide_folds;
  if (err) {
    if (log_level()) std::fprintf(stderr, "[tccl] copy-out allreduce failed: %s\n", cudaGetErrorString((cudaError_t)err));
    return tcclCudaError;
  }
  return tcclSuccess;
}

// Reduce-scatter on the copy-out engine: no copies, one launch of the
// register-load fold with P jobs, shard j of every send buffer folded into
// rank j's receive buffer. Needs every send and receive buffer to share its
// address mod 16 and the shard size to be a multiple of 16 bytes (so every
// shard starts at that same alignment); returns tcclInvalidUsage otherwise,
// and the caller takes the bulk engine.
tcclResult_t run_copy_out_reduce_scatter(tcclGroup* g, const void* const* send, void* const* recv,
                                         size_t rc, int dtype, int op, int es, cudaStream_t stream,
                                         int cap) {
  const int P = g->nranks;
  if (!register_fold_ok(kReduceScatter, P, mod16_of(P, send).data(),
                        mod16_of(P, (const void* const*)recv).data(), rc, es, 0))
    return tcclInvalidUsage;
  AnchorArgs aa;
  reduce_scatter_args(&aa, P, send, recv, rc, es);
  aa.sm_mask = sm_record_slot(g);
  aa.mixed_bf16 = mixed_bf16_fold();
  const uint64_t per_cta = (uint64_t)kAnchorThreads * anchor_vectors_per_thread(P, aa.wide != 0, dtype);
  uint64_t grid = std::max<uint64_t>(1, (aa.nvec * P + per_cta - 1) / per_cta);
  grid = std::min<uint64_t>(grid, cap > 0 ? (uint64_t)cap : (uint64_t)g->dev.sm_count);
  const int err = launch_anchor_reduce(dtype, op, aa, (int)grid, cap <= 0, stream);
  std::memset(&g->last, 0, sizeof(g->last));
  g->last.engine = kEngineCopyOut;
  g->last.store_mode = kStoreVec;
  g->last.ctas = (int)grid;
  g->last.threads = kAnchorThreads;
  g->last.ce_segments = 1;
  g->last.ce_wide_folds = aa.wide;
  if (err) {
    if (log_level()) std::fprintf(stderr, "[tccl] copy-out reduce-scatter failed: %s\n", cudaGetErrorString((cudaError_t)err));
    return tcclCudaError;
  }
  return tcclSuccess;
}

// All-gather on the copy-out engine: P x P (P x (P-1) in place) device-to-
// device copies spread over the group's copy streams. No kernel, no SM.
tcclResult_t run_copy_out_allgather(tcclGroup* g, const void* const* send, void* const* recv,
                                    size_t count, int es, cudaStream_t stream) {
  const int P = g->nranks;
  tcclResult_t r = ensure_ce_resources(g, 0);
  if (r != tcclSuccess) return r;
  const int used = std::min(g->cfg.ce_streams, P * P);
  const size_t bytes = count * (size_t)es;
  int err = cudaEventRecord(g->ce_fork_event, stream);
  for (int j = 0; j < used && !err; ++j) err = cudaStreamWaitEvent(g->ce_streams[j], g->ce_fork_event, 0);
  int j = 0, copies = 0;
  for (int q = 0; q < P && !err; ++q) {
    for (int k = 0; k < P && !err; ++k) {
      char* dst = static_cast<char*>(recv[k]) + (size_t)q * bytes;
      if (dst == static_cast<const char*>(send[q])) continue;  // in place: already there
      err = cudaMemcpyAsync(dst, send[q], bytes, cudaMemcpyDeviceToDevice, g->ce_streams[j]);
      j = (j + 1) % used;
      ++copies;
    }
  }
  const int jerr = join_ce_streams(g, used, stream);
  if (!err) err = jerr;
  std::memset(&g->last, 0, sizeof(g->last));
  g->last.engine = kEngineCopyOut;
  g->last.ce_copies = copies;
  if (err) {
    if (log_level()) std::fprintf(stderr, "[tccl] copy-out all-gather failed: %s\n", cudaGetErrorString((cudaError_t)err));
    return tcclCudaError;
  }
  return tcclSuccess;
}

}  // namespace tccl
