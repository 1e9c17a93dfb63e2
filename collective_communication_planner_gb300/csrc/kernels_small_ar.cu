// Warp / vec (small-message) engine instances for one collective.
#include "dispatch.cuh"

namespace tccl {

using namespace dev;

int launch_small_ar(int dtype, int op, int engine, int size_class, const void* args,
                    const LaunchShape& s, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  (void)op;
  TCCL_REDUCE_SWITCH(kAllReduce, launch_small_sc, engine, size_class, args, s, st)
}

}  // namespace tccl
