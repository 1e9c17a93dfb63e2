// M-to-N reshard kernel: strided row copies, each source piece read once and
// written to every destination replica of its block (load once, store to all).
#include "dispatch.cuh"
#include "reshard.h"

namespace tccl {
namespace {

__global__ void __launch_bounds__(256) reshard_kernel(const __grid_constant__ ReshardArgs a) {
  // an early (programmatic dependent) launch waits here for the stream's
  // previous kernel before any global access
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) dev::record_sm(a.sm_mask);
  const int lane = threadIdx.x & 31;
  const uint64_t nunits = a.unit_prefix[a.nwin];
  const uint64_t warp = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
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

}  // namespace

int launch_reshard(const ReshardArgs& a, int grid, bool early, void* stream) {
  LaunchShape s;
  s.grid = grid;
  s.threads = 256;
  s.smem = 0;
  s.early_launch = early ? 1 : 0;
  return dev::launch_maybe_early(reshard_kernel, a, s, static_cast<cudaStream_t>(stream));
}

}  // namespace tccl
