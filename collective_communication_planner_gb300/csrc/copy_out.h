// Copy-out engine: the kernel that folds P ranks with plain register loads
// (128-bit, or 256-bit where every buffer is 32-byte aligned past the head;
// no shared-memory staging), into one anchor rank's buffer before the
// GPU's copy engines fan the result out to the other ranks, or for a
// reduce-scatter into each shard's owner.
#pragma once

#include "internal.h"

namespace tccl {

constexpr int kAnchorThreads = 1024;

// One launch of the register-load fold: `njobs` independent folds of the P
// sources. Job j reads every p.src[r] from byte offset j * job_src_stride and
// writes p.dst[j]: one job (the copy-out allreduce segment, into the anchor's
// receive buffer) or P jobs (a reduce-scatter, shard j into rank j's receive
// buffer). Every source and destination of a job shares its address mod 16:
// `head_bytes` element-wise bytes, then `nvec` 16-byte vectors, then
// `tail_bytes` element-wise bytes, the same for every job.
struct AnchorArgs {
  BasePtrs<kMaxRanks> p;
  uint32_t* sm_mask;      // SM recorder bitmap or null
  uint64_t head_bytes;
  uint64_t nvec;
  uint64_t tail_bytes;
  uint64_t job_src_stride;
  int njobs;
  int nranks;
  int prefetch_first;  // set by the launcher for early launches: warm L2 before the wait
  int mixed_bf16;      // bf16 sums: fold with the mixed-precision add (same bits, fewer instructions)
  int wide;            // 256-bit loads (P = 2 to 8 or a multiple of 4; see anchor_wide_ok)
};

// 32-byte vectors each thread folds at a time with 256-bit loads: two for
// P = 2 with 4-byte types, one otherwise.
constexpr int anchor_wide_vectors(int nranks, int dtype) {
  return (nranks == 2 && dtype != kBF16) ? 2 : 1;
}
// 16-byte vectors each thread folds at a time: two for P = 2 and 4, one
// otherwise; with 256-bit loads, twice anchor_wide_vectors.
int anchor_vectors_per_thread(int nranks, bool wide = false, int dtype = kBF16);
// Whether a fold can take 256-bit loads: P = 2 to 8 or a multiple of 4, and every source and
// destination of every job 32-byte aligned once the head is skipped.
// TCCL_ANCHOR_WIDE=0 turns them off (the same bits either way).
bool anchor_wide_ok(const AnchorArgs& a);
// The register fold's arguments (rank count, jobs, pointers, head / vectors /
// tail split and the 256-bit choice; not sm_mask or mixed_bf16) for one
// allreduce segment, elements [off, off + n) of every send buffer into the
// anchor's receive buffer, all sharing the anchor's address mod 16 ...
void allreduce_segment_args(AnchorArgs* a, int nranks, const void* const* send,
                            void* anchor_recv, size_t off, size_t n, int es);
// ... and for a reduce-scatter, shard j of every send buffer into recv[j]
// (rc elements each, every buffer sharing recv[0]'s address mod 16).
void reduce_scatter_args(AnchorArgs* a, int nranks, const void* const* send,
                         void* const* recv, size_t rc, int es);
// early: programmatic dependent launch (uncapped calls only: a capped call
// must not hold SMs beyond its cap while it waits)
int launch_anchor_reduce(int dtype, int op, const AnchorArgs& a, int grid, bool early,
                         void* stream);

}  // namespace tccl
