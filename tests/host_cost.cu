// Host cost of one tcclAllReduce call, measured from C++ with no Python in
// the way: the decode-sized messages of the tensor-parallel workload (P = 8,
// bf16 [tokens, 8192] with 1, 8 and 64 tokens) and the small end of the fp32
// in-place sweep (4 KiB and 64 KiB per rank).
//
// For every case it prints one JSON line:
//   host_us        wall time per call of the enqueue loop (batches of 100
//                  calls, the device synchronised between batches, so the
//                  launch queue never fills and the time is the host's own);
//   device_us      CUDA-event time per call over back-to-back plain calls;
//   graph_us       CUDA-event time per call replaying a graph of 20 calls;
//   launch_us, launch_early_us  the same enqueue timing for an empty kernel
//                  launched plainly and with programmatic stream
//                  serialisation (the attribute the library's uncapped
//                  launches carry): the floor a library call cannot go under;
//   ok             every rank's result equals the exact sum P (P + 1) / 2 of
//                  the small integers 1..P each rank holds.
// Build: nvcc -gencode arch=compute_103a,code=sm_103a -O2 -I include
//        tests/host_cost.cu -o host_cost -L <package dir> -ltccl
#include <cuda_runtime.h>

#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "tccl.h"

namespace {

__global__ void empty_kernel() {}

__global__ void fill_bf16(unsigned short* p, size_t n, unsigned short v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = v;
}

__global__ void fill_f32(float* p, size_t n, float v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = v;
}

double now_us() {
  return std::chrono::duration<double, std::micro>(
             std::chrono::steady_clock::now().time_since_epoch())
      .count();
}

#define CK(x)                                                                  \
  do {                                                                         \
    cudaError_t e_ = (x);                                                      \
    if (e_ != cudaSuccess) {                                                   \
      std::fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
      return 2;                                                                \
    }                                                                          \
  } while (0)

#define TK(x)                                                                  \
  do {                                                                         \
    tcclResult_t r_ = (x);                                                     \
    if (r_ != tcclSuccess) {                                                   \
      std::fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, tcclGetErrorString(r_)); \
      return 3;                                                                \
    }                                                                          \
  } while (0)

struct Case {
  const char* name;
  tcclDataType_t dt;
  size_t count;
  bool in_place;
};

// Wall time per enqueue of fn(), in batches of 100 with a device sync between.
template <typename F>
double enqueue_us(F fn, cudaStream_t st, int batches) {
  double total = 0;
  for (int b = 0; b < batches + 2; ++b) {
    cudaStreamSynchronize(st);
    const double t0 = now_us();
    for (int i = 0; i < 100; ++i) fn();
    const double t1 = now_us();
    if (b >= 2) total += t1 - t0;  // the first two batches warm up
  }
  cudaStreamSynchronize(st);
  return total / (batches * 100.0);
}

}  // namespace

int main(int argc, char** argv) {
  const int P = 8;
  const int batches = argc > 1 ? std::atoi(argv[1]) : 50;
  const Case cases[] = {
      {"C5 [1, 8192] bf16 sum, out of place", tcclBfloat16, 8192, false},
      {"C5 [8, 8192] bf16 sum, out of place", tcclBfloat16, 8 * 8192, false},
      {"C5 [64, 8192] bf16 sum, out of place", tcclBfloat16, 64 * 8192, false},
      {"C3 4 KiB fp32 sum, in place", tcclFloat32, 1024, true},
      {"C3 64 KiB fp32 sum, in place", tcclFloat32, 16384, true},
  };
  CK(cudaSetDevice(0));
  cudaStream_t st;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  // the empty-launch floor, plain and with programmatic stream serialisation
  auto plain = [&] { empty_kernel<<<1, 32, 0, st>>>(); };
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(1);
  lc.blockDim = dim3(32);
  lc.stream = st;
  lc.attrs = attr;
  lc.numAttrs = 1;
  auto early = [&] { cudaLaunchKernelEx(&lc, empty_kernel); };
  const double launch_us = enqueue_us(plain, st, batches);
  const double launch_early_us = enqueue_us(early, st, batches);
  CK(cudaGetLastError());

  tcclGroup_t g;
  TK(tcclGroupCreate(P, &g));
  int failures = 0;
  for (const Case& c : cases) {
    const size_t es = c.dt == tcclBfloat16 ? 2 : 4;
    std::vector<void*> send(P), recv(P);
    for (int r = 0; r < P; ++r) {
      CK(cudaMalloc(&send[r], c.count * es));
      if (c.in_place) recv[r] = send[r];
      else CK(cudaMalloc(&recv[r], c.count * es));
    }
    // rank r holds r + 1 everywhere; before every timed block the inputs are
    // refilled, since in place the result overwrites them
    auto refill = [&]() -> int {
      for (int r = 0; r < P; ++r) {
        if (c.dt == tcclBfloat16) {
          float f = (float)(r + 1);
          unsigned int u;
          std::memcpy(&u, &f, 4);
          fill_bf16<<<64, 256, 0, st>>>((unsigned short*)send[r], c.count, (unsigned short)(u >> 16));
        } else {
          fill_f32<<<64, 256, 0, st>>>((float*)send[r], c.count, (float)(r + 1));
        }
      }
      CK(cudaStreamSynchronize(st));
      return 0;
    };
    auto call = [&] {
      tcclAllReduce(g, send.data(), recv.data(), c.count, c.dt, tcclSum, st, 0);
    };
    if (refill()) return 2;
    TK(tcclAllReduce(g, send.data(), recv.data(), c.count, c.dt, tcclSum, st, 0));  // plans
    CK(cudaStreamSynchronize(st));
    // correctness of one call
    bool ok = true;
    {
      std::vector<unsigned char> h(c.count * es);
      CK(cudaMemcpy(h.data(), recv[P - 1], h.size(), cudaMemcpyDeviceToHost));
      const float want = (float)(P * (P + 1) / 2);
      for (size_t i = 0; i < c.count && ok; ++i) {
        float v;
        if (c.dt == tcclBfloat16) {
          unsigned short b;
          std::memcpy(&b, &h[2 * i], 2);
          unsigned int u = (unsigned int)b << 16;
          std::memcpy(&v, &u, 4);
        } else {
          std::memcpy(&v, &h[4 * i], 4);
        }
        ok = v == want;
      }
    }
    if (c.in_place && refill()) return 2;
    const double host_us = enqueue_us(call, st, batches);
    CK(cudaGetLastError());
    // device time per call, back to back
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    const int reps = 2000;
    CK(cudaEventRecord(e0, st));
    for (int i = 0; i < reps; ++i) call();
    CK(cudaEventRecord(e1, st));
    CK(cudaEventSynchronize(e1));
    float ms = 0;
    CK(cudaEventElapsedTime(&ms, e0, e1));
    const double device_us = ms * 1e3 / reps;
    // graph of 20 calls, replayed
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    CK(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
    for (int i = 0; i < 20; ++i) call();
    CK(cudaStreamEndCapture(st, &graph));
    CK(cudaGraphInstantiate(&exec, graph, 0));
    for (int i = 0; i < 5; ++i) CK(cudaGraphLaunch(exec, st));
    const int greps = 200;
    CK(cudaEventRecord(e0, st));
    for (int i = 0; i < greps; ++i) CK(cudaGraphLaunch(exec, st));
    CK(cudaEventRecord(e1, st));
    CK(cudaEventSynchronize(e1));
    CK(cudaEventElapsedTime(&ms, e0, e1));
    const double graph_us = ms * 1e3 / (greps * 20.0);
    tcclResult_t async = tcclSuccess;
    TK(tcclGroupQueryError(g, &async));
    ok = ok && async == tcclSuccess;
    tcclLaunchInfo_t info;
    TK(tcclGetLastLaunchInfo(g, &info));
    std::printf("{\"mode\": \"host_cost\", \"case\": \"%s\", \"P\": %d, \"count\": %zu, "
                "\"bytes_per_rank\": %zu, \"engine\": %d, \"ctas\": %d, \"host_us\": %.3f, "
                "\"device_us\": %.3f, \"graph_us\": %.3f, \"launch_us\": %.3f, "
                "\"launch_early_us\": %.3f, \"ok\": %s}\n",
                c.name, P, c.count, c.count * es, info.engine, info.ctas, host_us, device_us,
                graph_us, launch_us, launch_early_us, ok ? "true" : "false");
    std::fflush(stdout);
    failures += ok ? 0 : 1;
    CK(cudaGraphExecDestroy(exec));
    CK(cudaGraphDestroy(graph));
    CK(cudaEventDestroy(e0));
    CK(cudaEventDestroy(e1));
    for (int r = 0; r < P; ++r) {
      CK(cudaFree(send[r]));
      if (!c.in_place) CK(cudaFree(recv[r]));
    }
  }
  TK(tcclGroupDestroy(g));
  CK(cudaStreamDestroy(st));
  return failures ? 1 : 0;
}
