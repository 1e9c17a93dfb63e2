// The register-load fold of the copy-out engine: P ranks folded into one
// anchor buffer (the allreduce's shard-in; the copy engines then do the
// other P-1 stores) or each shard into its owner (a reduce-scatter).
//
// Under a CTA cap the work of a few SMs decides the rate. Feeding a fold
// through TMA copies and shared memory costs each byte a shared-memory write
// and a read plus per-stage synchronisation, and a capped SM then reads about
// 50 GB/s; 128-bit register loads with eight in flight per thread read about
// 140 GB/s per SM on GB300, and 256-bit loads of the same bytes in flight
// (buffers 32-byte aligned) about 6% more. Every result goes to one buffer,
// so the kernel is read-bound.
#include <cstdlib>
#include <string>

#include "copy_out.h"
#include "dispatch.cuh"

namespace tccl {
namespace dev {
namespace {

// L2 policies: the inputs are read exactly once (evict first); the result is
// read back by the copy engines right after the kernel, up to P-1 times, and
// should still be in L2 then (evict last)
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// read-only path, no L1 allocation; HINT: with the L2 policy
template <bool HINT>
__device__ __forceinline__ uint4 ld_stream_v4(const void* p, uint64_t policy) {
  uint4 r;
  if (HINT)
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(policy));
  else
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
  return r;
}

template <bool HINT>
__device__ __forceinline__ void st_keep_v4(void* p, uint4 v, uint64_t policy) {
  if (HINT)
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
  else
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// 256-bit forms (sm_100 and later): one 32-byte vector as two 16-byte halves
__device__ __forceinline__ void ld_stream_v8(const void* p, uint64_t policy, uint4& lo, uint4& hi) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
      : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
      : "l"(p), "l"(policy));
}

__device__ __forceinline__ void st_keep_v8(void* p, uint4 lo, uint4 hi, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p),
               "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w),
               "l"(policy)
               : "memory");
}

// For each job, thread t of the grid folds vectors t, t + T, ... (T threads
// in all), U of them at a time. With the rank count fixed at compile time
// (NP = 2, 4, 8) every load of a step is issued before the first add;
// otherwise the ranks go in batches of 8 / U. Either way each accumulator receives the ranks in
// ascending order: the plain left fold over all P ranks.
// The fold of one vector: the streaming fold, or for bf16 sums with MIXED
// the mixed-precision adds (the same bits, fewer instructions).
template <int DT, int OP, bool MIXED>
struct AnchorFold {
  using type = typename StreamFold<DT, OP>::type;
};
template <>
struct AnchorFold<kBF16, kSum, true> {
  using type = MixedSumBF16;
};

// The job's unaligned head and tail (the bytes before and after its 16-byte
// vectors), one element per thread of the grid.
template <int DT, int OP>
__device__ __forceinline__ void anchor_edges(const AnchorArgs& a, int job, int P, uint32_t gtid) {
  constexpr int es = DT == kBF16 ? 2 : 4;
  const uint32_t nh = static_cast<uint32_t>(a.head_bytes / es);
  const uint32_t nt = static_cast<uint32_t>(a.tail_bytes / es);
  if (gtid >= nh + nt) return;
  Window w;
  w.src_sel = -1;
  w.dst_sel = static_cast<int16_t>(job);
  w.scalar = 1;
  w.task = 0;
  w.cta = -1;
  uint64_t e = gtid;
  const uint64_t job_off = static_cast<uint64_t>(job) * a.job_src_stride;
  if (gtid < nh) {
    w.src_off = job_off;
    w.dst_off = 0;
    w.bytes = static_cast<uint32_t>(a.head_bytes);
  } else {
    const uint64_t body_end = a.head_bytes + a.nvec * 16;
    w.src_off = job_off + body_end;
    w.dst_off = body_end;
    w.bytes = static_cast<uint32_t>(a.tail_bytes);
    e -= nh;
  }
  scalar_element<kAllReduce, DT, OP, kMaxRanks>(a.p, P, w, e);
}

template <int DT, int OP, int NP, int U, bool MIXED>
__global__ void __launch_bounds__(kAnchorThreads, 1) anchor_reduce_kernel(const __grid_constant__ AnchorArgs a) {
  constexpr int RB = NP > 0 ? NP : 8 / U;
  const int P = NP > 0 ? NP : a.nranks;
  // a job covers fewer than 2^28 vectors (register_fold_ok keeps larger ones
  // off this kernel), so vector indices and byte offsets within it fit 32 bits
  const uint32_t nthr = gridDim.x * blockDim.x;
  const uint32_t gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t nvec = static_cast<uint32_t>(a.nvec);
  // an early (programmatic dependent) launch gets here while the stream's
  // previous kernel may still run: it first warms L2 with the block's first
  // vectors of job 0 in every rank (a prefetch writes nothing, and L2 is
  // where every write lands, so nothing is read stale), then waits before
  // any global access
  if (a.prefetch_first && threadIdx.x < static_cast<unsigned>(P)) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t vs = blockIdx.x * blockDim.x + u * nthr;
      if (vs < nvec)
        bulk_prefetch_l2(static_cast<const char*>(a.p.src[threadIdx.x]) + a.head_bytes + static_cast<uint64_t>(vs) * 16,
                         min(blockDim.x, nvec - vs) * 16u);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) record_sm(a.sm_mask);
  // the two policy registers fit beside one vector per thread (64 registers
  // at 1024 threads), not beside two
  constexpr bool kHint = U == 1;
  const uint64_t load_policy = kHint ? l2_policy_evict_first() : 0;
  const uint64_t store_policy = kHint ? l2_policy_evict_last() : 0;
  for (int job = 0; job < a.njobs; ++job) {
    const uint64_t src_off = static_cast<uint64_t>(job) * a.job_src_stride + a.head_bytes;
    char* dst = static_cast<char*>(a.p.dst[job]) + a.head_bytes;
    for (uint32_t base = gtid; base < nvec; base += nthr * U) {
      typename AnchorFold<DT, OP, MIXED>::type acc[U];
      for (int r0 = 0; r0 < P; r0 += RB) {
        uint4 x[U][RB];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint32_t v = base + u * nthr;
#pragma unroll
          for (int k = 0; k < RB; ++k)
            if (v < nvec && (NP > 0 || r0 + k < P))
              x[u][k] = ld_stream_v4<kHint>(static_cast<const char*>(a.p.src[r0 + k]) + src_off +
                                            static_cast<uint64_t>(v) * 16, load_policy);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (base + u * nthr >= nvec) continue;
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            if (NP == 0 && r0 + k >= P) break;
            if (r0 + k == 0) acc[u].init(x[u][k]);
            else acc[u].add(x[u][k]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t v = base + u * nthr;
        if (v < nvec) st_keep_v4<kHint>(dst + static_cast<uint64_t>(v) * 16, acc[u].out(), store_policy);
      }
    }
    anchor_edges<DT, OP>(a, job, P, gtid);
  }
}

// The same fold with 256-bit loads (P = 2 to 8, 16, or a multiple of 4 read
// at run time, NP = 0): each thread folds U 32-byte vectors of every rank at
// a time, the ranks in batches of four (P = 2 and 3: all at once; P = 6: two
// batches of three; P = 5 and 7: four, then the rest), so each thread keeps
// as many bytes in flight as the 128-bit form with half the load
// instructions (P = 2 with 4-byte types: U = 2, twice as many). The two
// 16-byte halves of a vector have one accumulator each and receive the ranks
// in ascending order, as above. Needs every source and the destination
// 32-byte aligned after the head (the launcher checks); an odd last 16-byte
// vector is folded by the grid's last thread.
template <int DT, int OP, int NP, int U, bool MIXED>
__global__ void __launch_bounds__(kAnchorThreads, 1) anchor_reduce_wide_kernel(const __grid_constant__ AnchorArgs a) {
  static_assert(NP == 0 || (NP >= 2 && NP <= 8) || NP == 16, "a batched rank count");
  constexpr int RB = NP == 2 ? 2 : (NP == 3 || NP == 6) ? 3 : 4;
  const int P = NP > 0 ? NP : a.nranks;
  const uint32_t nthr = gridDim.x * blockDim.x;
  const uint32_t gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t nvec = static_cast<uint32_t>(a.nvec);
  const uint32_t nwide = nvec / 2;
  if (a.prefetch_first && threadIdx.x < static_cast<unsigned>(P)) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t vs = blockIdx.x * blockDim.x + u * nthr;
      if (vs < nwide)
        bulk_prefetch_l2(static_cast<const char*>(a.p.src[threadIdx.x]) + a.head_bytes + static_cast<uint64_t>(vs) * 32,
                         min(blockDim.x, nwide - vs) * 32u);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) record_sm(a.sm_mask);
  const uint64_t load_policy = l2_policy_evict_first();
  const uint64_t store_policy = l2_policy_evict_last();
  using Acc = typename AnchorFold<DT, OP, MIXED>::type;
  for (int job = 0; job < a.njobs; ++job) {
    const uint64_t src_off = static_cast<uint64_t>(job) * a.job_src_stride + a.head_bytes;
    char* dst = static_cast<char*>(a.p.dst[job]) + a.head_bytes;
    for (uint32_t base = gtid; base < nwide; base += nthr * U) {
      Acc lo[U], hi[U];
#pragma unroll (NP > 0 ? (NP + RB - 1) / RB : 1)
      for (int r0 = 0; r0 < P; r0 += RB) {
        uint4 xl[U][RB], xh[U][RB];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint32_t v = base + u * nthr;
#pragma unroll
          for (int k = 0; k < RB; ++k)
            if (v < nwide && (NP == 0 || r0 + k < NP))
              ld_stream_v8(static_cast<const char*>(a.p.src[r0 + k]) + src_off + static_cast<uint64_t>(v) * 32,
                           load_policy, xl[u][k], xh[u][k]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (base + u * nthr >= nwide) continue;
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            if (NP > 0 && r0 + k >= NP) break;
            if (r0 + k == 0) {
              lo[u].init(xl[u][k]);
              hi[u].init(xh[u][k]);
            } else {
              lo[u].add(xl[u][k]);
              hi[u].add(xh[u][k]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t v = base + u * nthr;
        if (v < nwide) st_keep_v8(dst + static_cast<uint64_t>(v) * 32, lo[u].out(), hi[u].out(), store_policy);
      }
    }
    if ((nvec & 1) && gtid == nthr - 1) {
      const uint64_t last = static_cast<uint64_t>(nvec - 1) * 16;
      Acc acc;
      for (int k = 0; k < P; ++k) {
        const uint4 x = ld_stream_v4<true>(static_cast<const char*>(a.p.src[k]) + src_off + last, load_policy);
        if (k == 0) acc.init(x);
        else acc.add(x);
      }
      st_keep_v4<true>(dst + last, acc.out(), store_policy);
    }
    anchor_edges<DT, OP>(a, job, P, gtid);
  }
}

template <int C, int D, int O>
int launch_anchor_t(const AnchorArgs& args, int grid, bool early, cudaStream_t st) {
  AnchorArgs a = args;
  a.prefetch_first = early ? 1 : 0;  // an ordinary launch has nothing to overlap
  LaunchShape s;
  s.grid = grid;
  s.threads = kAnchorThreads;
  s.smem = 0;
  s.early_launch = early ? 1 : 0;
  constexpr bool kCanMix = D == kBF16 && O == kSum;
  if (a.wide) {
    // P = 2: two vectors per thread where the accumulators allow (bf16 sums
    // hold 16 fp32 accumulators per vector: one)
    constexpr int U2 = anchor_wide_vectors(2, D);
    if (kCanMix && a.mixed_bf16) {
      switch (a.nranks) {
        case 2: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 2, U2, kCanMix>, a, s, st);
        case 3: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 3, 1, kCanMix>, a, s, st);
        case 4: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 4, 1, kCanMix>, a, s, st);
        case 5: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 5, 1, kCanMix>, a, s, st);
        case 6: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 6, 1, kCanMix>, a, s, st);
        case 7: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 7, 1, kCanMix>, a, s, st);
        case 8: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 8, 1, kCanMix>, a, s, st);
        case 16: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 16, 1, kCanMix>, a, s, st);
        default: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 0, 1, kCanMix>, a, s, st);
      }
    }
    switch (a.nranks) {
      case 2: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 2, U2, false>, a, s, st);
      case 3: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 3, 1, false>, a, s, st);
      case 4: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 4, 1, false>, a, s, st);
      case 5: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 5, 1, false>, a, s, st);
      case 6: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 6, 1, false>, a, s, st);
      case 7: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 7, 1, false>, a, s, st);
      case 8: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 8, 1, false>, a, s, st);
      case 16: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 16, 1, false>, a, s, st);
      default: return launch_maybe_early(anchor_reduce_wide_kernel<D, O, 0, 1, false>, a, s, st);
    }
  }
  if (kCanMix && a.mixed_bf16) {
    switch (a.nranks) {
      case 2: return launch_maybe_early(anchor_reduce_kernel<D, O, 2, 2, kCanMix>, a, s, st);
      case 4: return launch_maybe_early(anchor_reduce_kernel<D, O, 4, 2, kCanMix>, a, s, st);
      case 8: return launch_maybe_early(anchor_reduce_kernel<D, O, 8, 1, kCanMix>, a, s, st);
      default: return launch_maybe_early(anchor_reduce_kernel<D, O, 0, 1, kCanMix>, a, s, st);
    }
  }
  switch (a.nranks) {
    case 2: return launch_maybe_early(anchor_reduce_kernel<D, O, 2, 2, false>, a, s, st);
    case 4: return launch_maybe_early(anchor_reduce_kernel<D, O, 4, 2, false>, a, s, st);
    case 8: return launch_maybe_early(anchor_reduce_kernel<D, O, 8, 1, false>, a, s, st);
    default:  // other rank counts: one vector per thread (two would spill)
      return launch_maybe_early(anchor_reduce_kernel<D, O, 0, 1, false>, a, s, st);
  }
}

}  // namespace
}  // namespace dev

int anchor_vectors_per_thread(int nranks, bool wide, int dtype) {
  if (wide) return 2 * anchor_wide_vectors(nranks, dtype);
  return (nranks == 2 || nranks == 4) ? 2 : 1;
}

bool anchor_wide_ok(const AnchorArgs& a) {
  static const bool enabled = [] {
    const char* e = std::getenv("TCCL_ANCHOR_WIDE");
    return !(e && std::string(e) == "0");
  }();
  const int P = a.nranks;
  if (!enabled || !((P >= 2 && P <= 8) || (P > 8 && P % 4 == 0))) return false;
  for (int j = 0; j < a.njobs; ++j) {
    const uint64_t off = static_cast<uint64_t>(j) * a.job_src_stride + a.head_bytes;
    for (int k = 0; k < a.nranks; ++k)
      if ((reinterpret_cast<uintptr_t>(a.p.src[k]) + off) % 32) return false;
    if ((reinterpret_cast<uintptr_t>(a.p.dst[j]) + a.head_bytes) % 32) return false;
  }
  return true;
}

int launch_anchor_reduce(int dtype, int op, const AnchorArgs& a, int grid, bool early,
                         void* stream) {
  using namespace dev;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TCCL_REDUCE_SWITCH(kAllReduce, launch_anchor_t, a, grid, early, st)
}

}  // namespace tccl
