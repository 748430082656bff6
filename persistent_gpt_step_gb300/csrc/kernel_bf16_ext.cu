// Instantiation of the persistent step kernel for the rotary-embedding /
// gated-MLP / tied-embedding model variant (bf16 operands on tcgen05).
#include "launch.h"
#include "megakernel.cuh"

namespace pgs {
const void* step_kernel_bf16_ext() { return (const void*)&gpt_step_kernel<__nv_bfloat16, true, true>; }
}  // namespace pgs
