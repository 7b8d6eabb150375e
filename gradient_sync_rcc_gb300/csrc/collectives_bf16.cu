// collectives_bf16.cu -- bf16 instantiations of the multi-pointer pass
// (fp32 arithmetic, one round-to-nearest-even per output element).
#include "collectives.cuh"

namespace rcc {
cudaError_t launch_multi_ptr_bf16(Red red, bool fast, int nseg, const MultiPtrArgs& a,
                                  cudaStream_t stream) {
  return mp::launch_typed<__nv_bfloat16>(red, fast, nseg, a, stream);
}
cudaError_t bulk_copy_timeouts_bf16(uint32_t* out) { return mp::bulk_copy_timeouts(out); }
}  // namespace rcc
