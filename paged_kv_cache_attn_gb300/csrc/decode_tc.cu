// tcgen05 kernel for 128-row shared-prefix tiles (not built yet: the plan
// routes every segment to the split-KV kernel while kTensorCoreKernel is off).
#include "device_common.cuh"

namespace pkv {
struct SplitParams;
cudaError_t launch_tile_items(const CUtensorMap&, const CUtensorMap&,
                              const SplitParams&, const WorkItem*, int, int,
                              cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace pkv
