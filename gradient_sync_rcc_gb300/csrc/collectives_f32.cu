// collectives_f32.cu -- fp32 instantiations of the multi-pointer pass.
#include "collectives.cuh"

namespace rcc {
cudaError_t launch_multi_ptr_f32(Red red, bool fast, int nseg, const MultiPtrArgs& a,
                                 cudaStream_t stream) {
  return mp::launch_typed<float>(red, fast, nseg, a, stream);
}
cudaError_t bulk_copy_timeouts_f32(uint32_t* out) { return mp::bulk_copy_timeouts(out); }
}  // namespace rcc
