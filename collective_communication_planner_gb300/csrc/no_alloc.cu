// tcclAllReduceNoAlloc: the bulk-engine allreduce for callers that cannot
// allocate GPU memory.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory manager (which owns every device allocation and forbids
// side allocations), allocator hooks and out-of-memory handlers, or processes
// whose device memory is fully reserved up front. tcclGroupCreate allocates a
// status word and per-plan window tables, so it is out of reach for them.
// This entry point needs no group: the bulk kernel's scratch (status word,
// per-CTA offsets and the window table) lives in one file-scope __device__
// array below, which every GPU that loads this library holds until the
// process exits. The caller passes only inputs and outputs.
//
// A kernel that gives up on a bounded wait records tcclDeviceTimeout in the
// array's status word, which stays set until a later call reads it: each
// call first asks, without waiting, whether the kernel of the previous call
// on the device has finished (an event recorded after it) and, if so, reads
// the word on a private stream. A recorded timeout makes that call return
// tcclDeviceTimeout without launching anything, and clears the word.
#include "tccl.h"

#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"
#include "plan.h"

namespace tccl {
namespace {

constexpr size_t kScratchBytes = TCCL_NO_ALLOC_SCRATCH_BYTES;
// Layout of the scratch array (byte offsets).
constexpr size_t kStatusOff = 0;                 // int status word (cleared once read)
constexpr size_t kSchedOff = 64;                 // two 8-byte scheduler words (cleared every call)
constexpr size_t kCtaOff = 256;                  // uint32_t per-CTA scalar-window offsets
constexpr size_t kPrefixOff = kCtaOff + 4 * (TCCL_NO_ALLOC_MAX_CTAS + 1 + 63);
constexpr size_t kMaxBody = 1023;                // body windows (chunk prefix entries - 1)
constexpr size_t kWinOff = kPrefixOff + 8 * (kMaxBody + 1);
constexpr size_t kMaxWindows = (kScratchBytes - kWinOff) / sizeof(Window);
static_assert(kPrefixOff % 256 == 0 && kWinOff % 256 == 0, "table alignment");
static_assert(kMaxWindows >= TCCL_NO_ALLOC_MAX_CTAS + 3 * kMaxRanks, "scratch too small");

// The scratch. Host code must not use this name as an address: on the host
// it is only a stand-in for the symbol. The device address comes from
// cudaGetSymbolAddress, taken once per device below.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kScratchBytes];

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_no_alloc_scratch
  DeviceDesc dev;
  cudaEvent_t done = nullptr;        // recorded after every launch
  cudaStream_t side = nullptr;       // reads and clears the status word
  bool unread = false;               // a launch whose status word was not read yet
};

constexpr int kMaxDevices = 64;
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

// Once per device, with that device current: resolve the scratch array's
// device address and read the limits the lowering needs.
int setup_device(int device, DeviceSetup** out) {
  if (device < 0 || device >= kMaxDevices) return tcclInvalidUsage;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& s = g_setup[device];
  if (!s.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_no_alloc_scratch) != cudaSuccess || ptr == nullptr)
      return tcclCudaError;
    if (cudaDeviceGetAttribute(&s.dev.sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.dev.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.dev.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess)
      return tcclCudaError;
    if (prepare_bulk_kernels((size_t)s.dev.smem_optin) != 0) return tcclCudaError;
    if (!s.done && cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess)
      return tcclCudaError;
    if (!s.side && cudaStreamCreateWithFlags(&s.side, cudaStreamNonBlocking) != cudaSuccess)
      return tcclCudaError;
    s.scratch = static_cast<unsigned char*>(ptr);
    s.ready = true;
  }
  *out = &s;
  return tcclSuccess;
}

bool log_on() {
  const char* e = std::getenv("TCCL_LOG");
  return e && std::atoi(e) > 0;
}

// Test hook for the timeout path: TCCL_NO_ALLOC_INJECT_TIMEOUT_MS > 0 makes
// the first CTA of each launch wait that long on a barrier nothing signals.
uint64_t injected_wait_ns() {
  const char* e = std::getenv("TCCL_NO_ALLOC_INJECT_TIMEOUT_MS");
  const double ms = e ? std::atof(e) : 0.0;
  return ms > 0 ? (uint64_t)(ms * 1e6) : 0;
}

// The status of earlier launches, if the last one has finished: tcclSuccess
// (also while it is still running: it is read by a later call), or
// tcclDeviceTimeout, which is cleared here.
int read_status(DeviceSetup* ds) {
  if (!ds->unread) return tcclSuccess;
  const cudaError_t q = cudaEventQuery(ds->done);
  if (q == cudaErrorNotReady) return tcclSuccess;
  if (q != cudaSuccess) return tcclCudaError;
  int st = 0;
  if (cudaMemcpyFromSymbolAsync(&st, g_no_alloc_scratch, sizeof(int), kStatusOff,
                                cudaMemcpyDeviceToHost, ds->side) != cudaSuccess ||
      cudaStreamSynchronize(ds->side) != cudaSuccess)
    return tcclCudaError;
  ds->unread = false;
  if (st == 0) return tcclSuccess;
  if (cudaMemsetAsync(ds->scratch + kStatusOff, 0, sizeof(int), ds->side) != cudaSuccess ||
      cudaStreamSynchronize(ds->side) != cudaSuccess)
    return tcclCudaError;
  return tcclDeviceTimeout;
}

}  // namespace
}  // namespace tccl

using namespace tccl;

extern "C" tcclResult_t tcclAllReduceNoAlloc(int nranks, const void* const sendbufs[],
                                             void* const recvbufs[], size_t count,
                                             tcclDataType_t datatype, tcclRedOp_t op,
                                             cudaStream_t stream, int cta_cap) {
  int v = validate_collective_args(kAllReduce, nranks, sendbufs, recvbufs, count, datatype, op);
  if (v != tcclSuccess) return (tcclResult_t)v;
  if (count == 0 || (nranks == 1 && sendbufs[0] == recvbufs[0])) return tcclSuccess;
  // each call stages its plan from host memory with an ordinary copy, which
  // a stream capture cannot hold: refuse a capturing stream up front
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return tcclCudaError;
  if (cs != cudaStreamCaptureStatusNone) return tcclInvalidUsage;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return tcclCudaError;
  DeviceSetup* ds = nullptr;
  int st = setup_device(device, &ds);
  if (st != tcclSuccess) return (tcclResult_t)st;
  st = read_status(ds);
  if (st != tcclSuccess) return (tcclResult_t)st;

  const int es = datatype == tcclBfloat16 ? 2 : 4;
  Plan pl = plan_collective(kAllReduce, nranks, count, es, op);
  uint8_t sm[kMaxRanks], rm[kMaxRanks];
  pl.in_place = true;
  for (int r = 0; r < nranks; ++r) {
    sm[r] = (uint8_t)((uintptr_t)sendbufs[r] & 15);
    rm[r] = (uint8_t)((uintptr_t)recvbufs[r] & 15);
    pl.in_place = pl.in_place && sendbufs[r] == recvbufs[r];
  }
  Config cfg;
  cfg.engine = kEngineBulk;
  Lowered low;
  std::string why;
  if (!lower_plan(pl, sm, rm, cfg, ds->dev, cta_cap, &low, &why)) return tcclInvalidUsage;
  if (low.shape.grid > TCCL_NO_ALLOC_MAX_CTAS || low.win.size() > kMaxWindows ||
      (size_t)low.nbody > kMaxBody) {
    if (log_on())
      std::fprintf(stderr,
                   "[tccl] tcclAllReduceNoAlloc: plan needs %d CTAs, %zu windows (%d bodies); "
                   "the static scratch holds at most %d CTAs, %zu windows, %zu bodies\n",
                   low.shape.grid, low.win.size(), low.nbody, TCCL_NO_ALLOC_MAX_CTAS,
                   kMaxWindows, kMaxBody);
    return tcclInvalidUsage;
  }

  // Stage this call's plan into the shared scratch, in stream order, and
  // clear the chunk scheduler's counters (the status word keeps whatever an
  // earlier launch recorded until a call reads it).
  unsigned char* base = ds->scratch;
  const size_t wbytes = low.win.size() * sizeof(Window);
  const size_t pbytes = low.chunk_prefix.size() * sizeof(uint64_t);
  const size_t cbytes = low.cta_first.size() * sizeof(uint32_t);
  if (cudaMemsetAsync(base + kSchedOff, 0, kCtaOff - kSchedOff, stream) != cudaSuccess ||
      cudaMemcpyAsync(base + kCtaOff, low.cta_first.data(), cbytes, cudaMemcpyHostToDevice,
                      stream) != cudaSuccess ||
      cudaMemcpyAsync(base + kPrefixOff, low.chunk_prefix.data(), pbytes,
                      cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      (wbytes && cudaMemcpyAsync(base + kWinOff, low.win.data(), wbytes, cudaMemcpyHostToDevice,
                                 stream) != cudaSuccess))
    return tcclCudaError;

  BulkArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    a.p.src[r] = sendbufs[r];
    a.p.dst[r] = recvbufs[r];
  }
  a.win = reinterpret_cast<const Window*>(base + kWinOff);
  a.chunk_prefix = reinterpret_cast<const uint64_t*>(base + kPrefixOff);
  a.cta_first = reinterpret_cast<const uint32_t*>(base + kCtaOff);
  a.total_chunks = low.total_chunks;
  a.chunks_per_cta = low.chunks_per_cta;
  a.nbody = low.nbody;
  a.sched = reinterpret_cast<unsigned long long*>(base + kSchedOff);
  a.order = low.shape.order;
  a.prefetch_chunks = low.shape.prefetch_chunks;
  a.rank_streamed = low.shape.rank_streamed;
  a.load_evict_first = low.shape.load_evict_first;
  a.status = reinterpret_cast<int*>(base + kStatusOff);
  a.sm_mask = nullptr;
  a.timeout_ns = (uint64_t)(resolve_config(cfg).wait_timeout_ms * 1e6);
  a.inject_timeout_ns = injected_wait_ns();
  a.nranks = nranks;
  a.chunk_bytes = low.shape.chunk_bytes;
  a.stages = low.shape.stages;
  a.store_mode = low.shape.store_mode;
  a.consumer_warps = low.shape.consumer_warps;
  a.release_lag = low.shape.release_lag;
  a.elem_size = es;
  int err = launch_bulk(kAllReduce, datatype, op, a, low.shape, stream);
  if (err == 0) err = cudaEventRecord(ds->done, stream);
  if (err != 0) return tcclCudaError;
  ds->unread = true;
  return tcclSuccess;
}
