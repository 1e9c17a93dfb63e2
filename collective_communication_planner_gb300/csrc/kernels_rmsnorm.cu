// Allreduce of [rows, hidden] activations fused with an RMSNorm of each
// reduced row, before the row is stored to every rank (the Device API example
// the "NCCL Roadmap" post describes: receive, sum, normalise, send out in one
// kernel). The reduced row never leaves the chip unnormalised.
#include <cooperative_groups.h>

#include "dispatch.cuh"
#include "rmsnorm.h"

namespace tccl {
namespace {

// V: 16-byte vectors of a row per thread. Loads of RB ranks are issued
// together before they are folded (ascending rank order is kept), so a row
// costs a few memory round trips, not P of them. CTA b reduces row b first;
// with a.claim set (more rows than CTAs) it then claims rows from a device
// counter, so SMs that stream faster take more rows and the grid ends within
// about one row's time of itself; without it, rows b + G, b + 2G, ... One
// block barrier per row: the sums of squares of the warps are exchanged
// through a double-buffered slot, and every warp adds them up in the same
// order, so every warp derives the same scale.
template <int DT, int V>
__global__ void __launch_bounds__(kRmsMaxThreads) rmsnorm_kernel(const __grid_constant__ RmsArgs a) {
  using dev::Fold;
  constexpr int kVecElems = DT == kBF16 ? 8 : 4;
  constexpr int RB = 16 / V;  // ranks per load batch: V * RB 16-byte registers in flight
  extern __shared__ __align__(16) uint4 gamma_smem[];
  __shared__ float partial[2][kRmsMaxThreads / 32];
  __shared__ unsigned long long next_row[2];
  const uint32_t row_bytes = a.hidden * (DT == kBF16 ? 2u : 4u);
  // an early (programmatic dependent) launch gets here while the stream's
  // previous kernel may still run: when every CTA has one row and all of
  // them fit well inside L2, it first warms L2 with its row of every rank (a
  // prefetch writes nothing and L2 is where every write lands, so nothing is
  // read stale), then waits before any global access. GB300, P=8, 8192
  // bf16: 512 rows 25.5 -> 21.5 us; with more rows than CTAs the prefetched
  // first rows only crowd L2 (2048 rows: 83.2 -> 85.1 us without this bound)
  if (threadIdx.x < a.nranks && blockIdx.x < a.rows && a.rows <= gridDim.x &&
      a.rows * a.nranks * static_cast<uint64_t>(row_bytes) <= (static_cast<uint64_t>(64) << 20))
    dev::bulk_prefetch_l2(static_cast<const char*>(a.p.src[threadIdx.x]) + blockIdx.x * static_cast<uint64_t>(row_bytes),
                          row_bytes);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) dev::record_sm(a.sm_mask);
  const int P = a.nranks;
  const uint32_t nvec = a.hidden / kVecElems;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (uint32_t v = threadIdx.x; v < nvec; v += blockDim.x)
    gamma_smem[v] = dev::ld_global_v4(static_cast<const char*>(a.gamma) + v * 16ull);
  __syncthreads();
  int buf = 0;
  for (uint64_t t = blockIdx.x; t < a.rows; buf ^= 1) {
    // the row after this one: claimed now, its value needed (and published
    // through shared memory) only at this row's barrier, so the claim's round
    // trip overlaps the row's loads
    unsigned long long nxt = 0;
    if (threadIdx.x == 0) nxt = a.claim ? gridDim.x + atomicAdd(a.claim, 1ull) : t + gridDim.x;
    const uint64_t row_off = t * static_cast<uint64_t>(a.hidden) * (DT == kBF16 ? 2 : 4);
    Fold<DT, kSum> acc[V];
    for (int r0 = 0; r0 < P; r0 += RB) {
      uint4 x[V][RB];
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const uint32_t v = threadIdx.x + j * blockDim.x;
#pragma unroll
        for (int k = 0; k < RB; ++k)
          if (v < nvec && r0 + k < P)
            x[j][k] = dev::ld_global_v4(static_cast<const char*>(a.p.src[r0 + k]) + row_off + v * 16ull);
      }
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const uint32_t v = threadIdx.x + j * blockDim.x;
        if (v < nvec) {
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            if (r0 + k >= P) break;
            if (r0 + k == 0) acc[j].init(x[j][k]);
            else acc[j].add(x[j][k]);
          }
        }
      }
    }
    // sum of squares of the reduced row
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint32_t v = threadIdx.x + j * blockDim.x;
      if (v < nvec)
#pragma unroll
        for (int e = 0; e < kVecElems; ++e) ss = __fadd_rn(ss, __fmul_rn(acc[j].a[e], acc[j].a[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, o));
    if (lane == 0) partial[buf][warp] = ss;
    if (threadIdx.x == 0) next_row[buf] = nxt;
    // the one barrier of the row; a slot is written again two rows later,
    // after the next row's barrier, which every thread reaches only once it
    // has read this row's slot
    __syncthreads();
    float w = lane < nwarps ? partial[buf][lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = __fadd_rn(w, __shfl_xor_sync(0xFFFFFFFFu, w, o));
    const float scale = rsqrtf(__fadd_rn(__fdiv_rn(w, static_cast<float>(a.hidden)), a.eps));
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint32_t v = threadIdx.x + j * blockDim.x;
      if (v < nvec) {
        Fold<DT, kSum> g;
        g.init(gamma_smem[v]);
#pragma unroll
        for (int e = 0; e < kVecElems; ++e)
          acc[j].a[e] = __fmul_rn(__fmul_rn(acc[j].a[e], scale), g.a[e]);
        const uint4 y = acc[j].out();
        const uint64_t o = row_off + v * 16ull;
        for (int d = 0; d < P; ++d) dev::st_global_v4(static_cast<char*>(a.p.dst[d]) + o, y);
      }
    }
    t = next_row[buf];
  }
  // the last CTA to finish resets the counter for the next launch (every
  // CTA made its last claim before it counts itself finished)
  if (a.claim && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.claim + 1, 1ull) == gridDim.x - 1) {
      atomicExch(a.claim, 0ull);
      atomicExch(a.claim + 1, 0ull);
    }
  }
}

// Few rows (decode-sized calls): a cluster of kRmsCluster CTAs shares each
// row. CTA q of the cluster reduces and normalises a contiguous slice. Thread
// 0 of every CTA writes its slice's sum of squares into slot q of every CTA's
// shared memory (distributed shared memory), and after one cluster barrier
// each CTA adds its own slots in cluster-rank order, so every CTA derives the
// same scale. No CTA reads another's shared memory, so none waits for the
// others before it moves on or exits; the slots alternate between two sets
// from row to row, since a CTA may write the next row's sum while another
// still adds up this row's.
//
// V vectors per thread, RB ranks per load batch: a slice of at most one
// vector per thread takes V = 1 and RB = 8, so up to eight ranks cost one
// memory round trip, and loads its gamma vector once, before the first row,
// so the scale step waits on no load (with V = 4 the gamma vectors would cost
// the registers of a second resident CTA per SM; they are loaded after the
// scale).
template <int DT, int V, int RB>
__global__ void __launch_bounds__(kRmsClusterThreads)
    rmsnorm_cluster_kernel(const __grid_constant__ RmsArgs a) {
  namespace cg = cooperative_groups;
  using dev::Fold;
  constexpr int kVecElems = DT == kBF16 ? 8 : 4;
  __shared__ float partial[kRmsClusterThreads / 32];
  __shared__ float slots[2][kRmsCluster];
  cg::cluster_group cluster = cg::this_cluster();
  const int q = static_cast<int>(cluster.block_rank());
  const int C = static_cast<int>(cluster.num_blocks());
  const int P = a.nranks;
  const uint32_t nvec = a.hidden / kVecElems;
  const uint32_t per = (nvec + C - 1) / C;
  const uint32_t v0 = q * per;
  const uint32_t v1 = min(nvec, v0 + per);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const uint64_t cid = blockIdx.x / C;
  const uint64_t nclusters = gridDim.x / C;
  // as in rmsnorm_kernel: warm L2 with this CTA's slice of its first row of
  // every rank, then wait for the previous kernel before any global access
  if (threadIdx.x < P && cid < a.rows && v1 > v0)
    dev::bulk_prefetch_l2(static_cast<const char*>(a.p.src[threadIdx.x]) +
                              cid * static_cast<uint64_t>(a.hidden) * (DT == kBF16 ? 2 : 4) + v0 * 16ull,
                          (v1 - v0) * 16u);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) dev::record_sm(a.sm_mask);
  constexpr bool kGammaFirst = V == 1;
  Fold<DT, kSum> gam[V];
  if (kGammaFirst) {
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint32_t v = v0 + threadIdx.x + j * blockDim.x;
      if (v < v1) gam[j].init(dev::ld_global_v4(static_cast<const char*>(a.gamma) + v * 16ull));
    }
  }
  int buf = 0;
  for (uint64_t t = cid; t < a.rows; t += nclusters, buf ^= 1) {
    const uint64_t row_off = t * static_cast<uint64_t>(a.hidden) * (DT == kBF16 ? 2 : 4);
    Fold<DT, kSum> acc[V];
    for (int r0 = 0; r0 < P; r0 += RB) {
      uint4 x[V][RB];
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const uint32_t v = v0 + threadIdx.x + j * blockDim.x;
#pragma unroll
        for (int k = 0; k < RB; ++k)
          if (v < v1 && r0 + k < P)
            x[j][k] = dev::ld_global_v4(static_cast<const char*>(a.p.src[r0 + k]) + row_off + v * 16ull);
      }
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const uint32_t v = v0 + threadIdx.x + j * blockDim.x;
        if (v < v1) {
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            if (r0 + k >= P) break;
            if (r0 + k == 0) acc[j].init(x[j][k]);
            else acc[j].add(x[j][k]);
          }
        }
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint32_t v = v0 + threadIdx.x + j * blockDim.x;
      if (v < v1)
#pragma unroll
        for (int e = 0; e < kVecElems; ++e) ss = __fadd_rn(ss, __fmul_rn(acc[j].a[e], acc[j].a[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, o));
    if (lane == 0) partial[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float w = 0.f;
      for (int i = 0; i < nwarps; ++i) w = __fadd_rn(w, partial[i]);
      for (int i = 0; i < C; ++i) *cluster.map_shared_rank(&slots[buf][q], i) = w;
    }
    cluster.sync();  // every slice's sum of squares is in every CTA's slots
    float total = 0.f;
    for (int i = 0; i < C; ++i) total = __fadd_rn(total, slots[buf][i]);
    const float scale = rsqrtf(__fadd_rn(__fdiv_rn(total, static_cast<float>(a.hidden)), a.eps));
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint32_t v = v0 + threadIdx.x + j * blockDim.x;
      if (v < v1) {
        if (!kGammaFirst) gam[j].init(dev::ld_global_v4(static_cast<const char*>(a.gamma) + v * 16ull));
#pragma unroll
        for (int e = 0; e < kVecElems; ++e)
          acc[j].a[e] = __fmul_rn(__fmul_rn(acc[j].a[e], scale), gam[j].a[e]);
        const uint4 y = acc[j].out();
        const uint64_t o = row_off + v * 16ull;
        for (int d = 0; d < P; ++d) dev::st_global_v4(static_cast<char*>(a.p.dst[d]) + o, y);
      }
    }
  }
}

}  // namespace

int launch_rmsnorm_cluster(int dtype, const RmsArgs& a, int clusters, int cluster_size,
                           bool early, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * cluster_size));
  cfg.blockDim = dim3(kRmsClusterThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 2 : 1;
  // a slice of at most one vector per thread: one batch of up to 8 ranks
  const uint32_t nvec = a.hidden / (dtype == kBF16 ? 8u : 4u);
  const bool one = (nvec + cluster_size - 1) / cluster_size <= static_cast<uint32_t>(kRmsClusterThreads);
  cudaError_t e;
  if (dtype == kBF16)
    e = one ? cudaLaunchKernelEx(&cfg, rmsnorm_cluster_kernel<kBF16, 1, 8>, a)
            : cudaLaunchKernelEx(&cfg, rmsnorm_cluster_kernel<kBF16, 4, 4>, a);
  else
    e = one ? cudaLaunchKernelEx(&cfg, rmsnorm_cluster_kernel<kF32, 1, 8>, a)
            : cudaLaunchKernelEx(&cfg, rmsnorm_cluster_kernel<kF32, 4, 4>, a);
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

int launch_rmsnorm(int dtype, const RmsArgs& a, int grid, int threads, int vectors, bool early,
                   void* stream) {
  LaunchShape s;
  s.grid = grid;
  s.threads = threads;
  s.smem = static_cast<size_t>(a.hidden) * (dtype == kBF16 ? 2 : 4);
  s.early_launch = early ? 1 : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == kBF16)
    return vectors <= 4 ? dev::launch_maybe_early(rmsnorm_kernel<kBF16, 4>, a, s, st)
                        : dev::launch_maybe_early(rmsnorm_kernel<kBF16, 8>, a, s, st);
  return vectors <= 4 ? dev::launch_maybe_early(rmsnorm_kernel<kF32, 4>, a, s, st)
                      : dev::launch_maybe_early(rmsnorm_kernel<kF32, 8>, a, s, st);
}

int rmsnorm_ctas_per_sm(int dtype, int threads, int vectors, size_t smem) {
  int n = 0;
  cudaError_t e;
  if (dtype == kBF16)
    e = vectors <= 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rmsnorm_kernel<kBF16, 4>, threads, smem)
                     : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rmsnorm_kernel<kBF16, 8>, threads, smem);
  else
    e = vectors <= 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rmsnorm_kernel<kF32, 4>, threads, smem)
                     : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rmsnorm_kernel<kF32, 8>, threads, smem);
  return e == cudaSuccess ? n : 0;
}

}  // namespace tccl
