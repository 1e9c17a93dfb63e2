// M-to-N reshard kernel: strided row copies, each source piece read once and
// written to every destination replica of its block (load once, store to all).
#include "dispatch.cuh"
#include "reshard.h"

namespace tccl {
namespace {

__global__ void __launch_bounds__(256) reshard_kernel(const __grid_constant__ ReshardArgs a) {
  const int lane = threadIdx.x & 31;
  const uint64_t nunits = a.unit_prefix[a.nwin];  // the host's upload, no kernel's output
  const uint64_t warp = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
  // an early (programmatic dependent) launch gets here while the stream's
  // previous kernel may still run: each warp first warms L2 with its first
  // row segment (a prefetch writes nothing, and L2 is where every write
  // lands), then waits before any access to the buffers
  if (lane == 0 && warp < nunits) {
    const int wi = dev::find_window<0>(a.unit_prefix, a.nwin, warp);
    const ReshardWindow& w = a.win[wi];
    if (!w.scalar) {
      const uint64_t k = warp - a.unit_prefix[wi];
      const uint64_t segs = (w.bytes + kReshardSegBytes - 1) / kReshardSegBytes;
      const uint64_t row = k / segs;
      const uint32_t begin = static_cast<uint32_t>(k - row * segs) * kReshardSegBytes;
      dev::bulk_prefetch_l2(static_cast<const char*>(a.src[w.src]) + w.src_off + row * w.src_pitch + begin,
                            min(kReshardSegBytes, w.bytes - begin));
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) dev::record_sm(a.sm_mask);
  for (uint64_t u = warp; u < nunits; u += nwarps) {
    const int wi = dev::find_window<0>(a.unit_prefix, a.nwin, u);
    const ReshardWindow w = a.win[wi];
    const uint64_t k = u - a.unit_prefix[wi];
    const char* src = static_cast<const char*>(a.src[w.src]) + w.src_off;
    if (!w.scalar) {
      const uint64_t segs = (w.bytes + kReshardSegBytes - 1) / kReshardSegBytes;
      const uint64_t row = k / segs;
      const uint32_t begin = static_cast<uint32_t>(k - row * segs) * kReshardSegBytes;
      const uint32_t end = min(begin + kReshardSegBytes, w.bytes);
      const char* s = src + row * w.src_pitch;
      const uint64_t doff = w.dst_off + row * w.dst_pitch;
      // every load of the segment first (up to 8 per lane), then the stores:
      // a row piece costs one load latency, not one per 512 bytes
      constexpr int kPerLane = kReshardSegBytes / (32 * 16);
      uint4 v[kPerLane];
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const uint32_t b = begin + (lane + 32u * i) * 16u;
        if (b < end) v[i] = dev::ld_global_v4(s + b);
      }
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const uint32_t b = begin + (lane + 32u * i) * 16u;
        if (b < end) {
          uint64_t m = w.dst_mask;
          while (m) {
            const int d = __ffsll(static_cast<long long>(m)) - 1;
            m &= m - 1;
            dev::st_global_v4(static_cast<char*>(a.dst[d]) + doff + b, v[i]);
          }
        }
      }
    } else {
      const uint32_t es = static_cast<uint32_t>(a.elem_size);
      const uint32_t nel = w.bytes / es;
      const uint64_t segs = (nel + kReshardSegElems - 1) / kReshardSegElems;
      const uint64_t row = k / segs;
      const uint32_t begin = static_cast<uint32_t>(k - row * segs) * kReshardSegElems;
      const uint32_t end = min(begin + kReshardSegElems, nel);
      const char* s = src + row * w.src_pitch;
      const uint64_t doff = w.dst_off + row * w.dst_pitch;
      for (uint32_t e = begin + lane; e < end; e += 32) {
        uint64_t m = w.dst_mask;
        if (es == 2) {
          const uint16_t v = *reinterpret_cast<const uint16_t*>(s + e * 2ull);
          while (m) {
            const int d = __ffsll(static_cast<long long>(m)) - 1;
            m &= m - 1;
            *reinterpret_cast<uint16_t*>(static_cast<char*>(a.dst[d]) + doff + e * 2ull) = v;
          }
        } else {
          const uint32_t v = *reinterpret_cast<const uint32_t*>(s + e * 4ull);
          while (m) {
            const int d = __ffsll(static_cast<long long>(m)) - 1;
            m &= m - 1;
            *reinterpret_cast<uint32_t*>(static_cast<char*>(a.dst[d]) + doff + e * 4ull) = v;
          }
        }
      }
    }
  }
}

constexpr uint32_t kNoUnit = 0xFFFFFFFFu;

struct ReshardRingHead {
  uint64_t full[kReshardBulkStages];   // a stage's loads have landed
  uint64_t empty[kReshardBulkStages];  // a stage's stores have read it
  uint64_t never;                      // test hook: a barrier nothing completes
  uint32_t unit_win[kReshardBulkStages];
  BulkUnit unit[kReshardBulkStages];
  int abort_flag;
};
static_assert(sizeof(ReshardRingHead) <= kReshardBulkHeadBytes, "ring head");

__device__ __forceinline__ BulkUnit decode_bulk_unit(const ReshardWindow& w, uint64_t k) {
  constexpr uint32_t seg = kReshardBulkSegBytes;
  BulkUnit u;
  if (w.bytes >= seg) {  // one segment of one row
    const uint32_t segs = (w.bytes + seg - 1) / seg;
    u.row = static_cast<uint32_t>(k / segs);
    u.rows = 1;
    u.begin = static_cast<uint32_t>(k - static_cast<uint64_t>(u.row) * segs) * seg;
    u.n = min(seg, w.bytes - u.begin);
  } else {  // whole rows, as many as fit in a stage
    const uint32_t per = seg / w.bytes;
    u.row = static_cast<uint32_t>(k) * per;
    u.rows = min(per, w.nrows - u.row);
    u.begin = 0;
    u.n = w.bytes;
  }
  return u;
}

// The bulk engine: a persistent CTA streams work units through a ring of
// shared-memory stages. Thread 0 takes units (each CTA's first
// kReshardBulkStages fixed, the rest claimed from a counter) and loads each
// with cp.async.bulk; thread 32 stores every staged unit to each destination
// replica with bulk stores and frees the stage once those have read it. A
// unit is read from memory once whatever the number of replicas. Every wait
// is bounded: a wait that runs out flags the CTA's abort, records a timeout
// in the status word, and both threads leave after their copies in flight
// have finished with shared memory.
__global__ void __launch_bounds__(kReshardBulkThreads, 1)
    reshard_bulk_kernel(const __grid_constant__ ReshardArgs a) {
  using namespace dev;
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int S = kReshardBulkStages;
  constexpr uint32_t seg = kReshardBulkSegBytes;
  ReshardRingHead& h = *reinterpret_cast<ReshardRingHead*>(smem);
  unsigned char* ring = smem + kReshardBulkHeadBytes;
  volatile int* abort_flag = &h.abort_flag;
  if (threadIdx.x == 0) {
    for (int k = 0; k < S; ++k) {
      mbar_init(&h.full[k], 1);
      mbar_init(&h.empty[k], 1);
    }
    mbar_init(&h.never, 1);
    h.abort_flag = 0;
    fence_mbar_init();
  }
  const uint64_t nunits = a.unit_prefix[a.nwin];  // the host's upload, no kernel's output
  // an early (programmatic dependent) launch gets here while the stream's
  // previous kernel may still run: thread 0 first warms L2 with this CTA's
  // fixed first units (a prefetch writes nothing, and L2 is where every
  // write lands, so nothing is read stale), then all wait before any access
  // to the buffers
  if (threadIdx.x == 0) {
    for (int j = 0; j < S; ++j) {
      const uint64_t u = blockIdx.x + static_cast<uint64_t>(j) * gridDim.x;
      if (u >= nunits) break;
      const int wi = find_window<0>(a.unit_prefix, a.nwin, u);
      const ReshardWindow& w = a.win[wi];
      const BulkUnit bu = decode_bulk_unit(w, u - a.unit_prefix[wi]);
      const char* src = static_cast<const char*>(a.src[w.src]) + w.src_off +
                        static_cast<uint64_t>(bu.row) * w.src_pitch + bu.begin;
      for (uint32_t r = 0; r < min(bu.rows, 8u); ++r)  // a few rows of a unit of short ones
        bulk_prefetch_l2(src + static_cast<uint64_t>(r) * w.src_pitch, bu.n);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) record_sm(a.sm_mask);
  __syncthreads();
  if ((threadIdx.x & 31) != 0) return;

  if (threadIdx.x == 0) {
    const uint64_t grid = gridDim.x;
    const uint64_t claimed_base = static_cast<uint64_t>(S) * grid;
    uint32_t taken = 0;
    unsigned long long next_claim = claimed_base + atomicAdd(&a.sched[0], 1ull);
    uint32_t it = 0;
    bool ok = true;
    for (;; ++it) {
      uint64_t u;
      if (taken < static_cast<uint32_t>(S)) {
        u = blockIdx.x + static_cast<uint64_t>(taken) * grid;
        ++taken;
      } else {
        u = next_claim;
        if (u < nunits) next_claim = claimed_base + atomicAdd(&a.sched[0], 1ull);
      }
      const uint32_t k = it % S;
      if (it >= static_cast<uint32_t>(S)) {
        ok = wait_bounded(&h.empty[k], ((it / S) & 1) ^ 1, abort_flag, a.timeout_ns, a.status, true);
        if (!ok) break;
      }
      if (u >= nunits) {
        h.unit_win[k] = kNoUnit;  // published by the arrive's release
        mbar_arrive(&h.full[k]);
        break;
      }
      const int wi = find_window<0>(a.unit_prefix, a.nwin, u);
      const ReshardWindow& w = a.win[wi];
      const BulkUnit bu = decode_bulk_unit(w, u - a.unit_prefix[wi]);
      h.unit_win[k] = static_cast<uint32_t>(wi);
      h.unit[k] = bu;
      mbar_arrive_expect_tx(&h.full[k], bu.n * bu.rows);
      const char* src = static_cast<const char*>(a.src[w.src]) + w.src_off +
                        static_cast<uint64_t>(bu.row) * w.src_pitch + bu.begin;
      unsigned char* st = ring + static_cast<size_t>(k) * seg;
      for (uint32_t r = 0; r < bu.rows; ++r)
        bulk_load(st + static_cast<size_t>(r) * bu.n, src + static_cast<uint64_t>(r) * w.src_pitch, bu.n,
                  &h.full[k]);
    }
    if (!ok) {
      // an abort: let every load issued land before shared memory goes away
      // (only the last S iterations can be in flight)
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t j = first; j < it; ++j)
        wait_bounded(&h.full[j % S], (j / S) & 1, abort_flag, a.timeout_ns, a.status, false);
    }
    // the last CTA to finish claiming resets the counter for the next launch
    __threadfence();
    if (atomicAdd(&a.sched[1], 1ull) == grid - 1) {
      atomicExch(&a.sched[0], 0ull);
      atomicExch(&a.sched[1], 0ull);
    }
    return;
  }
  if (threadIdx.x != 32) return;
  // stores: up to kReshardBulkLag stages' stores in flight, the rest of the
  // ring left for loads
  constexpr int lag = kReshardBulkLag;
  for (uint32_t it = 0;; ++it) {
    const uint32_t k = it % S;
    bool ok = wait_bounded(&h.full[k], (it / S) & 1, abort_flag, a.timeout_ns, a.status, true);
    if (ok && a.inject_timeout_ns && blockIdx.x == 0 && it == 0)
      ok = wait_bounded(&h.never, 0, abort_flag, a.inject_timeout_ns, a.status, true);
    if (!ok) break;
    const uint32_t wi = h.unit_win[k];
    if (wi == kNoUnit) break;
    const ReshardWindow& w = a.win[wi];
    const BulkUnit bu = h.unit[k];
    const unsigned char* st = ring + static_cast<size_t>(k) * seg;
    const uint64_t doff = w.dst_off + static_cast<uint64_t>(bu.row) * w.dst_pitch + bu.begin;
    fence_proxy_async_smem();
    for (uint32_t r = 0; r < bu.rows; ++r) {
      uint64_t m = w.dst_mask;
      while (m) {
        const int d = __ffsll(static_cast<long long>(m)) - 1;
        m &= m - 1;
        bulk_store(static_cast<char*>(a.dst[d]) + doff + static_cast<uint64_t>(r) * w.dst_pitch,
                   st + static_cast<size_t>(r) * bu.n, bu.n);
      }
    }
    bulk_commit();
    bulk_wait_read<lag>();
    if (it >= static_cast<uint32_t>(lag)) mbar_arrive(&h.empty[(it - lag) % S]);
  }
  // leave once the stores have read shared memory; the grid's completion
  // makes their writes visible
  bulk_wait_read<0>();
}

}  // namespace

int prepare_reshard_kernels(size_t smem_bytes) {
  const size_t want = kReshardBulkHeadBytes + (size_t)kReshardBulkStages * kReshardBulkSegBytes;
  if (smem_bytes < want) return 0;  // the planner then keeps every reshard on the warp kernel
  return static_cast<int>(cudaFuncSetAttribute(reshard_bulk_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(want)));
}

int launch_reshard_bulk(const ReshardArgs& a, int grid, size_t smem, bool early, void* stream) {
  LaunchShape s;
  s.grid = grid;
  s.threads = kReshardBulkThreads;
  s.smem = smem;
  s.early_launch = early ? 1 : 0;
  return dev::launch_maybe_early(reshard_bulk_kernel, a, s, static_cast<cudaStream_t>(stream));
}

int launch_reshard(const ReshardArgs& a, int grid, bool early, void* stream) {
  LaunchShape s;
  s.grid = grid;
  s.threads = 256;
  s.smem = 0;
  s.early_launch = early ? 1 : 0;
  return dev::launch_maybe_early(reshard_kernel, a, s, static_cast<cudaStream_t>(stream));
}

}  // namespace tccl
