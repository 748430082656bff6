// Instantiation of the persistent step kernel for bf16 operands on tcgen05.
#include "launch.h"
#include "megakernel.cuh"

namespace pgs {
const void* step_kernel_bf16() { return (const void*)&gpt_step_kernel<__nv_bfloat16, true>; }
}  // namespace pgs
