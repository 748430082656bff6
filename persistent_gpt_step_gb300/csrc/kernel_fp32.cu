// Instantiation of the persistent step kernel for the fp32 (SIMT) arithmetic.
#include "launch.h"
#include "megakernel.cuh"

namespace pgs {
const void* step_kernel_fp32() { return (const void*)&gpt_step_kernel<float, false>; }
}  // namespace pgs
