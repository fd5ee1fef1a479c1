// Table of compiled router kernel variants (one per element type and row layout).
#pragma once

#include <stddef.h>

namespace moe {

struct RouterVariant {
  int LPR, VW, NV;         // lanes per row, elements per vector, vectors per lane
  const void* fwd;         // persistent kernel, forward phases
  const void* step;        // persistent kernel, forward + dispatch + backward
  const void* bwd;         // streaming backward kernel
};

// Variants compiled for bf16 / fp32 logits; *n receives the count.
const RouterVariant* router_variants_bf16(int* n);
const RouterVariant* router_variants_fp32(int* n);
// The dispatch-only persistent kernel.
const void* dispatch_kernel();

}  // namespace moe
