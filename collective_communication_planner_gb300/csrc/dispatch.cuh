// Launch helpers: map runtime (dtype, op, engine, size class) onto kernel
// template instances.
#pragma once

#include "kernels_common.cuh"

namespace tccl {
namespace dev {

template <int C, int D, int O>
int launch_bulk_t(const BulkArgs& a, const LaunchShape& s, cudaStream_t st);

template <int C, int D, int O>
int launch_reduce_t(const BulkArgs& a, const LaunchShape& s, cudaStream_t st) {
  reduce_kernel<C, D, O><<<s.grid, s.threads, s.smem, st>>>(a);
  return static_cast<int>(cudaGetLastError());
}

template <int C, int D, int O>
int set_reduce_smem(size_t bytes) {
  return static_cast<int>(cudaFuncSetAttribute(reduce_kernel<C, D, O>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(bytes)));
}

// (dtype, op) -> F<C, D, O> for the pairs the TMA-reduce engine supports
#define TCCL_TMA_REDUCE_SWITCH(COLL, FN, ...)                               \
  switch (dtype * 3 + op) {                                                 \
    case kF32 * 3 + kSum: return FN<COLL, kF32, kSum>(__VA_ARGS__);         \
    case kBF16 * 3 + kMin: return FN<COLL, kBF16, kMin>(__VA_ARGS__);       \
    case kBF16 * 3 + kMax: return FN<COLL, kBF16, kMax>(__VA_ARGS__);       \
    case kI32 * 3 + kSum: return FN<COLL, kI32, kSum>(__VA_ARGS__);         \
    case kI32 * 3 + kMin: return FN<COLL, kI32, kMin>(__VA_ARGS__);         \
    case kI32 * 3 + kMax: return FN<COLL, kI32, kMax>(__VA_ARGS__);         \
    default: return static_cast<int>(cudaErrorInvalidValue);                \
  }

template <int C, int D, int O>
int set_bulk_smem(size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(bulk_kernel<C, D, O>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bulk_kernel<C, D, O>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  return static_cast<int>(e);
}

// `kernel<<<…>>>(args)` or, with s.early_launch, the same launch with
// programmatic stream serialisation (the kernel waits in
// griddepcontrol.wait before touching global memory)
template <typename Kernel, typename Args>
int launch_maybe_early(Kernel kernel, const Args& a, const LaunchShape& s, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(s.threads));
  cfg.dynamicSmemBytes = s.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = s.early_launch ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a);
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

// bulk engine: an uncapped launch starts early (its CTAs take each SM as the
// previous kernel's CTA there exits); a capped one is an ordinary launch
template <int C, int D, int O>
int launch_bulk_t(const BulkArgs& a, const LaunchShape& s, cudaStream_t st) {
  return launch_maybe_early(bulk_kernel<C, D, O>, a, s, st);
}

template <int C, int D, int O, int MAXR, int MAXW, bool SHFL>
int launch_small_np(const SmallArgs<MAXR, MAXW>& a, const LaunchShape& s, cudaStream_t st) {
  // rank counts up to 8 compiled in (small tables), and 16 (large tables:
  // graph-captured on GB300, P = 16 at 16-512 KiB per rank, the vec engine
  // went from 4.2-5.1 to 2.2-3.3 us and the warp engine from 2.7-12 to
  // 2.2-10 us)
  if constexpr (MAXR == kSmallRanks) {
    switch (a.nranks) {
      case 2: return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 2>, a, s, st);
      case 3: return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 3>, a, s, st);
      case 4: return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 4>, a, s, st);
      case 5: return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 5>, a, s, st);
      case 6: return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 6>, a, s, st);
      case 7: return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 7>, a, s, st);
      case 8: return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 8>, a, s, st);
      default: break;
    }
  }
  if constexpr (MAXR != kSmallRanks) {
    if (a.nranks == 16) return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 16>, a, s, st);
  }
  return launch_maybe_early(small_kernel<C, D, O, MAXR, MAXW, SHFL, 0>, a, s, st);
}

template <int C, int D, int O, int MAXR, int MAXW>
int launch_small_t(int engine, const void* args, const LaunchShape& s, cudaStream_t st) {
  const auto& a = *static_cast<const SmallArgs<MAXR, MAXW>*>(args);
  if (engine == kEngineWarp) return launch_small_np<C, D, O, MAXR, MAXW, true>(a, s, st);
  return launch_small_np<C, D, O, MAXR, MAXW, false>(a, s, st);
}

template <int C, int D, int O>
int launch_small_sc(int engine, int size_class, const void* args, const LaunchShape& s,
                    cudaStream_t st) {
  if (size_class == 0) return launch_small_t<C, D, O, kSmallRanks, kSmallWindows>(engine, args, s, st);
  return launch_small_t<C, D, O, kMaxRanks, kLargeWindows>(engine, args, s, st);
}

// (dtype, op) -> F<C, D, O>(args...) for reducing collectives
#define TCCL_REDUCE_SWITCH(COLL, FN, ...)                                   \
  switch (dtype * 3 + op) {                                                 \
    case kF32 * 3 + kSum: return FN<COLL, kF32, kSum>(__VA_ARGS__);         \
    case kF32 * 3 + kMin: return FN<COLL, kF32, kMin>(__VA_ARGS__);         \
    case kF32 * 3 + kMax: return FN<COLL, kF32, kMax>(__VA_ARGS__);         \
    case kBF16 * 3 + kSum: return FN<COLL, kBF16, kSum>(__VA_ARGS__);       \
    case kBF16 * 3 + kMin: return FN<COLL, kBF16, kMin>(__VA_ARGS__);       \
    case kBF16 * 3 + kMax: return FN<COLL, kBF16, kMax>(__VA_ARGS__);       \
    case kI32 * 3 + kSum: return FN<COLL, kI32, kSum>(__VA_ARGS__);         \
    case kI32 * 3 + kMin: return FN<COLL, kI32, kMin>(__VA_ARGS__);         \
    case kI32 * 3 + kMax: return FN<COLL, kI32, kMax>(__VA_ARGS__);         \
    default: return static_cast<int>(cudaErrorInvalidValue);                \
  }

// all-gather only needs the element size
#define TCCL_COPY_SWITCH(FN, ...)                                                   \
  return (dtype == kBF16) ? FN<kAllGather, kBF16, kSum>(__VA_ARGS__)                \
                          : FN<kAllGather, kF32, kSum>(__VA_ARGS__);

}  // namespace dev
}  // namespace tccl
