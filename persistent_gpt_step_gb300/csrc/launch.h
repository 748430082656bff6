// launch.h — entry points of the compiled persistent kernels (one translation
// unit per arithmetic type).
#pragma once
#include "graph.h"

namespace pgs {
const void* step_kernel_fp32();  // SIMT, fp32 everywhere
const void* step_kernel_bf16();  // tcgen05 GEMMs, bf16 operands, fp32 accumulation
const void* step_kernel_bf16_ext();  // the same with rotary embedding and the gated MLP
}  // namespace pgs
