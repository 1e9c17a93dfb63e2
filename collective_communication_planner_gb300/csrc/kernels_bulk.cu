// Bulk (TMA pipeline) engine instances and launcher.
#include "dispatch.cuh"

namespace tccl {

using namespace dev;

int launch_bulk(int coll, int dtype, int op, const BulkArgs& a, const LaunchShape& s,
                void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (coll == kAllReduce) { TCCL_REDUCE_SWITCH(kAllReduce, launch_bulk_t, a, s, st) }
  if (coll == kReduceScatter) { TCCL_REDUCE_SWITCH(kReduceScatter, launch_bulk_t, a, s, st) }
  TCCL_COPY_SWITCH(launch_bulk_t, a, s, st)
}

int launch_reduce(int coll, int dtype, int op, const BulkArgs& a, const LaunchShape& s,
                  void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (coll == kAllReduce) { TCCL_TMA_REDUCE_SWITCH(kAllReduce, launch_reduce_t, a, s, st) }
  if (coll == kReduceScatter) { TCCL_TMA_REDUCE_SWITCH(kReduceScatter, launch_reduce_t, a, s, st) }
  return static_cast<int>(cudaErrorInvalidValue);
}

int prepare_bulk_kernels(size_t smem_bytes) {
  int err = 0;
  for (int dtype = 0; dtype < 3; ++dtype) {
    for (int op = 0; op < 3; ++op) {
      int e = [&]() -> int { TCCL_REDUCE_SWITCH(kAllReduce, set_bulk_smem, smem_bytes) }();
      if (e) err = e;
      e = [&]() -> int { TCCL_REDUCE_SWITCH(kReduceScatter, set_bulk_smem, smem_bytes) }();
      if (e) err = e;
    }
    int e = [&]() -> int { TCCL_COPY_SWITCH(set_bulk_smem, smem_bytes) }();
    if (e) err = e;
    for (int op = 0; op < 3; ++op) {
      if (!tma_reduce_supported(dtype, op)) continue;
      int r = [&]() -> int { TCCL_TMA_REDUCE_SWITCH(kAllReduce, set_reduce_smem, smem_bytes) }();
      if (r) err = r;
      r = [&]() -> int { TCCL_TMA_REDUCE_SWITCH(kReduceScatter, set_reduce_smem, smem_bytes) }();
      if (r) err = r;
    }
  }
  return err;
}

}  // namespace tccl
