// Table of compiled router kernel variants (one per element type and row layout).
#pragma once

#include <stddef.h>

namespace moe {

struct RouterVariant {
  int LPR, VW, NV;         // lanes per row, elements per vector, vectors per lane
  int NR;                  // row groups a consumer warp works on at once in the forward
  int staged;              // rows streamed through the shared-memory ring (16-byte rows)
  int min_blocks;          // CTAs per SM the persistent kernels are compiled for
  const void* fwd;         // persistent kernel, forward phases
  const void* step;        // persistent kernel, forward + dispatch + backward
  const void* bwd;         // streaming backward kernel
  const void* step_split;  // the step with the softmax sum and P formed in the backward (renormalised
                           // gates; bf16 rows of 32 lanes only, else null)
};

// Variants compiled for bf16 / fp32 logits; *n receives the count.
const RouterVariant* router_variants_bf16_staged(int* n);
const RouterVariant* router_variants_bf16_direct(int* n);
const RouterVariant* router_variants_fp32_staged(int* n);
const RouterVariant* router_variants_fp32_direct(int* n);
// The extended step (bias selection, masked P, gate gradients) of the same row
// layouts, in tables of their own (compiled in separate units).
struct StepExtVariant {
  int LPR, VW, NV, NR, staged, min_blocks;
  const void* step_ext;    // persistent kernel, the extended step
  const void* fwd_ext;     // persistent kernel, the extended step's forward alone (moe_router_fwd_ex)
};
const StepExtVariant* step_ext_bf16_staged(int* n);
const StepExtVariant* step_ext_bf16_direct(int* n);
const StepExtVariant* step_ext_fp32_staged(int* n);
const StepExtVariant* step_ext_fp32_direct(int* n);

// Kernels of the full backward, per row layout.  vec: 16-byte rows read VW
// elements per load.
struct ExtVariant {
  int LPR, VW, NV;
  int vec;
  const void* bwd;         // router_bwd_full_kernel
};
const ExtVariant* ext_variants_bf16(int* n);
const ExtVariant* ext_variants_fp32(int* n);

// The dispatch-only persistent kernel (compiled for kDispatchMinBlocks CTAs per SM).
const void* dispatch_kernel();
constexpr int kDispatchMinBlocks = 1;

}  // namespace moe
