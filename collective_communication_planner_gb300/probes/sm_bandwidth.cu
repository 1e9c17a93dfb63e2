// Per-SM memory bandwidth probe (measurement program, not part of the
// library). It bounds what a CTA cap can deliver: with G CTAs, a collective
// cannot move more than G times one SM's ceiling for its read/write mix.
//
// Each CTA streams its own contiguous region [cta * region, (cta + 1) * region)
// of two 2.5 GiB device buffers; region is a multiple of 64 KiB and
// grid * region never exceeds a buffer (checked before every launch). Every
// mbarrier wait is bounded by %globaltimer (0.5 s) and reports through an
// error word instead of hanging. Prints one JSON line per (probe, grid).
//
// Probes: 128-bit loads (read), 128-bit stores (write), load+store copy,
// cp.async.bulk loads into a shared-memory ring (read, per copy size), and
// bulk loads feeding 128-bit or bulk stores (copy, per copy size).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>

#define CK(x)                                                                        \
  do {                                                                               \
    cudaError_t e_ = (x);                                                            \
    if (e_ != cudaSuccess) {                                                         \
      std::printf("{\"error\": \"%s\", \"line\": %d}\n", cudaGetErrorString(e_), __LINE__); \
      std::exit(1);                                                                  \
    }                                                                                \
  } while (0)

namespace {

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(c) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t tx) {
  asm volatile("{ .reg .b64 s; mbarrier.arrive.expect_tx.shared::cta.b64 s, [%0], %1; }" ::"r"(
                   saddr(b)), "r"(tx)
               : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
  asm volatile("{ .reg .b64 s; mbarrier.arrive.shared::cta.b64 s, [%0]; }" ::"r"(saddr(b))
               : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t ph) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(ph)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ bool mb_wait(uint64_t* b, uint32_t ph, int* err, volatile int* abort_flag) {
  const uint64_t t0 = now_ns();
  for (uint32_t i = 0;; ++i) {
    if (mb_try(b, ph)) return true;
    if (*abort_flag) return false;
    if ((i & 31) == 0 && now_ns() - t0 > 500000000ull) {
      atomicExch(err, 1);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t n, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(saddr(dst)),
      "l"(src), "r"(n), "r"(saddr(bar))
      : "memory");
}

template <int U>
__global__ void __launch_bounds__(1024) read_ldg(const uint4* __restrict__ src, size_t rv,
                                                 uint32_t* sink) {
  const uint4* p = src + static_cast<size_t>(blockIdx.x) * rv;
  uint32_t acc = 0;
  for (size_t base = threadIdx.x; base < rv; base += static_cast<size_t>(blockDim.x) * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t i = base + static_cast<size_t>(u) * blockDim.x;
      v[u] = i < rv ? __ldcs(p + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  if (acc == 0x9E3779B9u) sink[blockIdx.x] = acc;  // keeps the loads alive
}

__global__ void __launch_bounds__(1024) write_stg(uint4* dst, size_t rv) {
  uint4* p = dst + static_cast<size_t>(blockIdx.x) * rv;
  const uint4 v = make_uint4(threadIdx.x, blockIdx.x, 1, 2);
  for (size_t i = threadIdx.x; i < rv; i += blockDim.x) __stcs(p + i, v);
}

template <int U>
__global__ void __launch_bounds__(1024) copy_ldg_stg(const uint4* __restrict__ src, uint4* dst,
                                                     size_t rv) {
  const uint4* s = src + static_cast<size_t>(blockIdx.x) * rv;
  uint4* d = dst + static_cast<size_t>(blockIdx.x) * rv;
  for (size_t base = threadIdx.x; base < rv; base += static_cast<size_t>(blockDim.x) * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t i = base + static_cast<size_t>(u) * blockDim.x;
      if (i < rv) v[u] = __ldcs(s + i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t i = base + static_cast<size_t>(u) * blockDim.x;
      if (i < rv) __stcs(d + i, v[u]);
    }
  }
}

// Bulk loads of `chunk` bytes into an S-stage ring. One producer thread; with
// `store_mode` 0 nobody uses the data (read probe), 1: consumer warps copy the
// stage out with 128-bit stores, 2: one thread issues a bulk store of the stage.
__global__ void __launch_bounds__(1024, 1) tma_pipe(const char* src, char* dst, size_t region,
                                                    uint32_t chunk, int S, int store_mode,
                                                    int* err) {
  extern __shared__ __align__(1024) unsigned char sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm);
  uint64_t* empty = full + 32;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + 32);
  unsigned char* ring = sm + 1024;
  const int cw = static_cast<int>(blockDim.x / 32) - 1;
  if (threadIdx.x == 0) {
    for (int k = 0; k < S; ++k) {
      mb_init(&full[k], 1);
      mb_init(&empty[k], store_mode == 1 ? cw : 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const char* s = src + static_cast<size_t>(blockIdx.x) * region;
  char* d = dst + static_cast<size_t>(blockIdx.x) * region;
  const uint32_t n = static_cast<uint32_t>(region / chunk);
  if (threadIdx.x < 32) {
    if (threadIdx.x != 0) return;
    uint32_t it = 0;
    for (; it < n; ++it) {
      const uint32_t k = it % S;
      if (it >= static_cast<uint32_t>(S)) {
        uint64_t* gate = store_mode == 0 ? &full[k] : &empty[k];
        const uint32_t ph = store_mode == 0 ? ((it / S) - 1) & 1 : ((it / S) & 1) ^ 1;
        if (!mb_wait(gate, ph, err, abort_flag)) break;
      }
      mb_expect(&full[k], chunk);
      bulk_load(ring + static_cast<size_t>(k) * chunk, s + static_cast<size_t>(it) * chunk, chunk,
                &full[k]);
    }
    const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
    for (uint32_t j = first; j < it; ++j) {
      const uint64_t t0 = now_ns();
      while (!mb_try(&full[j % S], (j / S) & 1) && now_ns() - t0 < 500000000ull) {
      }
    }
    return;
  }
  if (store_mode == 0) return;
  const int ct = threadIdx.x - 32;
  const int nct = cw * 32;
  if (store_mode == 2) {
    if (ct != 0) return;
    for (uint32_t it = 0; it < n; ++it) {
      const uint32_t k = it % S;
      if (!mb_wait(&full[k], (it / S) & 1, err, abort_flag)) break;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                       d + static_cast<size_t>(it) * chunk),
                   "r"(saddr(ring + static_cast<size_t>(k) * chunk)), "r"(chunk)
                   : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
      if (it >= 1) mb_arrive(&empty[(it - 1) % S]);
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    return;
  }
  for (uint32_t it = 0; it < n; ++it) {
    const uint32_t k = it % S;
    const bool ok = mb_wait(&full[k], (it / S) & 1, err, abort_flag);
    if (__any_sync(0xFFFFFFFFu, !ok)) break;
    const uint4* st = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(k) * chunk);
    uint4* dd = reinterpret_cast<uint4*>(d + static_cast<size_t>(it) * chunk);
    for (uint32_t v = ct; v < chunk / 16; v += nct) __stcs(dd + v, st[v]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mb_arrive(&empty[k]);
  }
}

}  // namespace

int main() {
  const size_t kBuf = static_cast<size_t>(2560) << 20;
  char *a, *b;
  uint32_t* sink;
  int* err;
  CK(cudaMalloc(&a, kBuf));
  CK(cudaMalloc(&b, kBuf));
  CK(cudaMalloc(&sink, 4096));
  CK(cudaMalloc(&err, 4));
  CK(cudaMemset(a, 1, kBuf));
  CK(cudaMemset(b, 0, kBuf));
  CK(cudaMemset(err, 0, 4));
  CK(cudaFuncSetAttribute(tma_pipe, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448));
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  int sm_count = 0;
  CK(cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, 0));
  const int grids[] = {1, 16, 32, sm_count};
  struct Tma {
    uint32_t chunk;
    int stages;
  };
  const Tma tma_shapes[] = {{8192, 24}, {16384, 13}, {32768, 6}, {65536, 3}};
  for (int g : grids) {
    const size_t region = (g <= 16 ? (static_cast<size_t>(128) << 20) : kBuf / g) & ~static_cast<size_t>(0xFFFF);
    if (region == 0 || static_cast<size_t>(g) * region > kBuf) return 1;
    const size_t rv = region / 16;
    auto time_it = [&](const char* probe, double bytes_per_region, auto&& launch) {
      launch();
      CK(cudaDeviceSynchronize());
      CK(cudaEventRecord(e0));
      launch();
      CK(cudaEventRecord(e1));
      CK(cudaEventSynchronize(e1));
      float ms = 0;
      CK(cudaEventElapsedTime(&ms, e0, e1));
      const double gbs = bytes_per_region * static_cast<double>(region) * g / (ms * 1e-3) / 1e9;
      std::printf("{\"probe\": \"%s\", \"grid\": %d, \"ms\": %.4f, \"GBps\": %.1f, \"GBps_per_sm\": %.1f}\n",
                  probe, g, ms, gbs, gbs / g);
      std::fflush(stdout);
    };
    time_it("read ldg.128 x16/thread", 1.0, [&] { read_ldg<16><<<g, 1024>>>(reinterpret_cast<const uint4*>(a), rv, sink); });
    time_it("write stg.128", 1.0, [&] { write_stg<<<g, 1024>>>(reinterpret_cast<uint4*>(b), rv); });
    time_it("copy ldg/stg.128 x8", 2.0, [&] { copy_ldg_stg<8><<<g, 1024>>>(reinterpret_cast<const uint4*>(a), reinterpret_cast<uint4*>(b), rv); });
    for (const Tma& t : tma_shapes) {
      const size_t smem = 1024 + static_cast<size_t>(t.stages) * t.chunk;
      if (smem > 232448 || t.stages > 32 || region % t.chunk) return 1;
      char name[96];
      std::snprintf(name, sizeof name, "read bulk %uK x%d", t.chunk >> 10, t.stages);
      time_it(name, 1.0, [&] { tma_pipe<<<g, 32, smem>>>(a, b, region, t.chunk, t.stages, 0, err); });
      std::snprintf(name, sizeof name, "copy bulk %uK x%d + stg.128 (16 warps)", t.chunk >> 10, t.stages);
      time_it(name, 2.0, [&] { tma_pipe<<<g, 544, smem>>>(a, b, region, t.chunk, t.stages, 1, err); });
      std::snprintf(name, sizeof name, "copy bulk %uK x%d + bulk store", t.chunk >> 10, t.stages);
      time_it(name, 2.0, [&] { tma_pipe<<<g, 64, smem>>>(a, b, region, t.chunk, t.stages, 2, err); });
    }
  }
  int h_err = 0;
  CK(cudaMemcpy(&h_err, err, 4, cudaMemcpyDeviceToHost));
  std::printf("{\"wait_timeouts\": %d}\n", h_err);
  return h_err ? 2 : 0;
}
