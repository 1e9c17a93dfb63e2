// Copy-engine probe: what the GPU's copy engines add to a CTA-capped
// allreduce. Prints one JSON line per measurement.
//
//  A. one device-to-device cudaMemcpyAsync of 1 GiB;
//  B. a 7-way fan-out of 128 MiB (7 x 128 MiB copies from one source), cut
//     into pieces of 2..128 MiB, spread over 1, 2, 4 or 7 streams;
//  C. a 1 GiB copy while a kernel holds every SM for 30 ms: if the copy ends
//     first, it used no SM;
//  D. the copy-out pipeline at a 16 or 32 CTA cap, P = 8, 128 MiB per rank:
//     per segment a register-load fold of 8 ranks into rank 0 (1024 threads
//     per CTA), then 7 copies of the segment from rank 0 to ranks 1..7 on 4
//     streams; timed with the copies, without them, and copies alone;
//  E. the host link: pinned host memory to the device and back, 512 MiB each
//     way, in 1, 2, 4 or 8 pieces on as many streams, one direction or both
//     at once.
//
// Every buffer is 128 MiB or 1 GiB; each index is checked against its buffer
// (segment offsets + segment sizes <= 128 MiB, fan-out destinations
// r * 128 MiB + 128 MiB <= 1 GiB). Every wait is bounded (the hold kernel
// stops after 30 ms of %globaltimer or 2^30 iterations).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#define CK(x)                                                                  \
  do {                                                                         \
    cudaError_t e_ = (x);                                                      \
    if (e_ != cudaSuccess) {                                                   \
      std::printf("{\"error\": \"%s\", \"line\": %d}\n", cudaGetErrorString(e_), __LINE__); \
      std::exit(1);                                                            \
    }                                                                          \
  } while (0)

namespace {

constexpr size_t kMiB = (size_t)1 << 20;
constexpr size_t kRank = 128 * kMiB;  // bytes per rank buffer
constexpr int kRanks = 8;

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void hold_kernel(uint64_t ns, uint32_t* sink) {
  extern __shared__ unsigned char smem[];
  const uint64_t t0 = now_ns();
  uint32_t i = 0;
  for (; i < (1u << 30); ++i)
    if ((i & 255) == 0 && now_ns() - t0 > ns) break;
  if (threadIdx.x == 0 && i == 12345u) sink[blockIdx.x] = smem[0];
}

struct Ranks {
  const uint4* src[kRanks];
  uint4* dst;
};

__device__ __forceinline__ uint4 load_nc(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// bf16 sum of 8 ranks in fp32, ascending rank order, one rounding
__global__ void __launch_bounds__(1024, 1) fold8(Ranks r, uint32_t nvec) {
  const uint32_t nthr = gridDim.x * blockDim.x;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += nthr) {
    uint4 x[kRanks];
#pragma unroll
    for (int k = 0; k < kRanks; ++k) x[k] = load_nc(r.src[k] + v);
    float acc[8];
#pragma unroll
    for (int k = 0; k < kRanks; ++k) {
      const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
        acc[2 * j] = k ? __fadd_rn(acc[2 * j], lo) : lo;
        acc[2 * j + 1] = k ? __fadd_rn(acc[2 * j + 1], hi) : hi;
      }
    }
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      out[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    r.dst[v] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

float elapsed(cudaEvent_t a, cudaEvent_t b) {
  float ms;
  CK(cudaEventElapsedTime(&ms, a, b));
  return ms;
}

}  // namespace

int main() {
  int sms = 0, engines = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  CK(cudaDeviceGetAttribute(&engines, cudaDevAttrAsyncEngineCount, 0));
  std::printf("{\"probe\": \"device\", \"sms\": %d, \"async_engines\": %d}\n", sms, engines);
  char *big_a, *big_b;
  CK(cudaMalloc(&big_a, 8 * kRank));
  CK(cudaMalloc(&big_b, 8 * kRank));
  CK(cudaMemset(big_a, 0x3c, 8 * kRank));
  CK(cudaMemset(big_b, 0, 8 * kRank));
  uint32_t* sink;
  CK(cudaMalloc(&sink, 4096));
  cudaStream_t st[8];
  for (int i = 0; i < 8; ++i) CK(cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking));
  cudaEvent_t e0, e1, ek, ev[8], seg_ev[64];
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  CK(cudaEventCreate(&ek));
  for (int i = 0; i < 8; ++i) CK(cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming));
  for (int i = 0; i < 64; ++i) CK(cudaEventCreateWithFlags(&seg_ev[i], cudaEventDisableTiming));

  // A
  float best = 1e9f;
  for (int rep = 0; rep < 3; ++rep) {
    CK(cudaEventRecord(e0, st[0]));
    CK(cudaMemcpyAsync(big_b, big_a, 8 * kRank, cudaMemcpyDeviceToDevice, st[0]));
    CK(cudaEventRecord(e1, st[0]));
    CK(cudaEventSynchronize(e1));
    const float ms = elapsed(e0, e1);
    if (ms < best) best = ms;
  }
  std::printf("{\"probe\": \"A one 1 GiB device-to-device copy\", \"ms\": %.4f, \"copy_GBps\": %.1f}\n",
              best, 8 * kRank / (best * 1e6));

  // B: source = first 128 MiB of big_a, destinations = big_b + r * 128 MiB
  for (size_t piece_mib : {2, 4, 8, 16, 32, 64, 128}) {
    for (int ns : {1, 2, 4, 7}) {
      const size_t piece = piece_mib * kMiB;
      const int npieces = (int)(kRank / piece);
      best = 1e9f;
      for (int rep = 0; rep < 2; ++rep) {
        CK(cudaDeviceSynchronize());
        CK(cudaEventRecord(e0, st[0]));
        for (int s = 1; s <= ns; ++s) CK(cudaStreamWaitEvent(st[s], e0, 0));
        int j = 0;
        for (int k = 0; k < npieces; ++k)
          for (int r = 0; r < 7; ++r) {
            CK(cudaMemcpyAsync(big_b + r * kRank + k * piece, big_a + k * piece, piece,
                               cudaMemcpyDeviceToDevice, st[1 + j]));
            j = (j + 1) % ns;
          }
        for (int s = 1; s <= ns; ++s) {
          CK(cudaEventRecord(ev[s], st[s]));
          CK(cudaStreamWaitEvent(st[0], ev[s], 0));
        }
        CK(cudaEventRecord(e1, st[0]));
        CK(cudaEventSynchronize(e1));
        const float ms = elapsed(e0, e1);
        if (ms < best) best = ms;
      }
      std::printf("{\"probe\": \"B 7-way fan-out of 128 MiB\", \"piece_mib\": %zu, \"streams\": %d, "
                  "\"ms\": %.4f, \"copy_GBps\": %.1f}\n",
                  piece_mib, ns, best, 7 * kRank / (best * 1e6));
    }
  }

  // C
  CK(cudaFuncSetAttribute(hold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
  CK(cudaDeviceSynchronize());
  CK(cudaEventRecord(e0, st[0]));
  hold_kernel<<<sms, 128, 200 * 1024, st[0]>>>(30000000ull, sink);
  CK(cudaGetLastError());
  CK(cudaEventRecord(ek, st[0]));
  CK(cudaStreamWaitEvent(st[1], e0, 0));
  CK(cudaMemcpyAsync(big_b, big_a, 8 * kRank, cudaMemcpyDeviceToDevice, st[1]));
  CK(cudaEventRecord(e1, st[1]));
  CK(cudaDeviceSynchronize());
  std::printf("{\"probe\": \"C 1 GiB copy beside a kernel holding every SM\", \"hold_ms\": %.3f, "
              "\"copy_done_ms\": %.3f}\n",
              elapsed(e0, ek), elapsed(e0, e1));

  // D: rank r's send buffer = big_a + r * 128 MiB, receive buffer = big_b + r * 128 MiB
  for (int cap : {16, 32}) {
    for (size_t seg_mib : {16, 32}) {
      for (int mode = 0; mode < 3; ++mode) {  // 0 folds only, 1 copies only, 2 both
        const size_t seg = seg_mib * kMiB;
        const int nseg = (int)(kRank / seg);
        best = 1e9f;
        for (int rep = 0; rep < 4; ++rep) {
          CK(cudaDeviceSynchronize());
          CK(cudaEventRecord(e0, st[0]));
          for (int k = 0; k < nseg; ++k) {
            const size_t off = k * seg;
            if (mode != 1) {
              Ranks rk;
              for (int r = 0; r < kRanks; ++r)
                rk.src[r] = reinterpret_cast<const uint4*>(big_a + r * kRank + off);
              rk.dst = reinterpret_cast<uint4*>(big_b + off);
              fold8<<<cap, 1024, 0, st[0]>>>(rk, (uint32_t)(seg / 16));
              CK(cudaGetLastError());
            }
            if (mode == 0) continue;
            CK(cudaEventRecord(seg_ev[k], st[0]));
            for (int j = 1; j <= 4; ++j) CK(cudaStreamWaitEvent(st[j], seg_ev[k], 0));
            for (int r = 1; r < kRanks; ++r)
              CK(cudaMemcpyAsync(big_b + r * kRank + off, big_b + off, seg, cudaMemcpyDeviceToDevice,
                                 st[1 + (r - 1) % 4]));
          }
          if (mode != 0)
            for (int j = 1; j <= 4; ++j) {
              CK(cudaEventRecord(ev[j], st[j]));
              CK(cudaStreamWaitEvent(st[0], ev[j], 0));
            }
          CK(cudaEventRecord(e1, st[0]));
          CK(cudaEventSynchronize(e1));
          const float ms = elapsed(e0, e1);
          if (ms < best) best = ms;
        }
        static const char* kMode[3] = {"folds only", "copies only", "folds and copies"};
        std::printf("{\"probe\": \"D copy-out pipeline P=8 128 MiB per rank\", \"cap\": %d, \"seg_mib\": %zu, "
                    "\"mode\": \"%s\", \"ms\": %.4f, \"alg_fraction_of_6.8TBps\": %.4f}\n",
                    cap, seg_mib, kMode[mode], best, 2.0 * kRanks * kRank / (best * 1e6) / 6800.0);
      }
    }
  }
  // E: host buffers of 512 MiB each way (pinned); device side = big_a / big_b
  {
    const size_t bytes = 4 * kRank;
    char *h_in, *h_out;
    CK(cudaMallocHost(&h_in, bytes));
    CK(cudaMallocHost(&h_out, bytes));
    std::memset(h_in, 1, bytes);
    std::memset(h_out, 0, bytes);
    for (int dir = 0; dir < 3; ++dir) {  // 0 host->device, 1 device->host, 2 both
      for (int ns : {1, 2, 4, 8}) {
        const size_t piece = bytes / ns;
        best = 1e9f;
        for (int rep = 0; rep < 3; ++rep) {
          CK(cudaDeviceSynchronize());
          CK(cudaEventRecord(e0, st[0]));
          for (int j = 0; j < 8; ++j) CK(cudaStreamWaitEvent(st[j], e0, 0));
          for (int k = 0; k < ns; ++k) {
            if (dir != 1)
              CK(cudaMemcpyAsync(big_a + k * piece, h_in + k * piece, piece, cudaMemcpyHostToDevice, st[k % 8]));
            if (dir != 0)
              CK(cudaMemcpyAsync(h_out + k * piece, big_b + k * piece, piece, cudaMemcpyDeviceToHost,
                                 st[(k + (dir == 2 ? 4 : 0)) % 8]));
          }
          for (int j = 1; j < 8; ++j) {
            CK(cudaEventRecord(ev[j], st[j]));
            CK(cudaStreamWaitEvent(st[0], ev[j], 0));
          }
          CK(cudaEventRecord(e1, st[0]));
          CK(cudaEventSynchronize(e1));
          const float ms = elapsed(e0, e1);
          if (ms < best) best = ms;
        }
        static const char* kDir[3] = {"host to device", "device to host", "both directions"};
        std::printf("{\"probe\": \"E host link, pinned, 512 MiB each way\", \"direction\": \"%s\", "
                    "\"pieces\": %d, \"ms\": %.4f, \"GBps_total\": %.1f}\n",
                    kDir[dir], ns, best, (dir == 2 ? 2.0 : 1.0) * bytes / (best * 1e6));
      }
    }
    CK(cudaFreeHost(h_in));
    CK(cudaFreeHost(h_out));
  }
  CK(cudaDeviceSynchronize());
  std::printf("{\"probe\": \"done\"}\n");
  return 0;
}
