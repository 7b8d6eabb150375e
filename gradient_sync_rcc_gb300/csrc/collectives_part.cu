// collectives_part.cu -- one unit of the multi-pointer pass: the kernels of one
// element type and one reduction.  The build compiles this file once per
// (RCC_PART_DT, RCC_PART_RED, RCC_PART_FAST) combination that the host
// dispatcher names (fp32 and bf16; rank-order sum, tree sum, max, min, copy),
// so the instantiations build in parallel instead of in one long unit.
#include "collectives.cuh"

#if !defined(RCC_PART_DT) || !defined(RCC_PART_RED) || !defined(RCC_PART_FAST)
#error "collectives_part.cu is built with -DRCC_PART_DT=.. -DRCC_PART_RED=.. -DRCC_PART_FAST=.."
#endif

namespace rcc {
namespace mp {
template cudaError_t launch_part<RCC_PART_DT, RCC_PART_RED, (RCC_PART_FAST != 0)>(
    int nseg, const MultiPtrArgs& a, cudaStream_t stream);
}  // namespace mp
}  // namespace rcc
