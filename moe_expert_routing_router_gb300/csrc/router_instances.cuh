// Explicit instantiation helpers for the router kernel variants.
#pragma once

#include "router_kernels.cuh"
#include "router_table.h"

namespace moe {
// The split step kernel of a variant, where it has one.
template <class DT, int LPR, int VW, int NV, int NR, bool STAGED, int MINB>
constexpr const void* split_step_kernel() {
  if constexpr (STAGED && kFastTopk<DT, LPR, VW, NV>)
    return reinterpret_cast<const void*>(&router_persistent_kernel<DT, LPR, VW, NV, NR, kModeStepSplit, STAGED, MINB>);
  else
    return nullptr;
}
}  // namespace moe

#define MOE_ROUTER_VARIANT(DT, LPR, VW, NV, NR, STAGED, MINB)                                                       \
  {LPR, VW, NV, NR, STAGED, MINB,                                                                                    \
   reinterpret_cast<const void*>(&::moe::router_persistent_kernel<DT, LPR, VW, NV, NR, ::moe::kModeFwd, STAGED, MINB>), \
   reinterpret_cast<const void*>(&::moe::router_persistent_kernel<DT, LPR, VW, NV, NR, ::moe::kModeStep, STAGED, MINB>), \
   reinterpret_cast<const void*>(&::moe::router_bwd_kernel<DT, LPR, VW, NV>),                                        \
   ::moe::split_step_kernel<DT, LPR, VW, NV, NR, STAGED, MINB>()}

#define MOE_ROUTER_VARIANT_ITEM(DT, LPR, VW, NV, NR, STAGED, MINB) MOE_ROUTER_VARIANT(DT, LPR, VW, NV, NR, STAGED, MINB),

#define MOE_STEP_EXT_VARIANT_ITEM(DT, LPR, VW, NV, NR, STAGED, MINB)                                                  \
  {LPR, VW, NV, NR, STAGED, MINB,                                                                                     \
   reinterpret_cast<const void*>(&::moe::router_persistent_kernel<DT, LPR, VW, NV, NR, ::moe::kModeStepExt, STAGED, MINB>), \
   reinterpret_cast<const void*>(&::moe::router_persistent_kernel<DT, LPR, VW, NV, NR, ::moe::kModeFwdExt, STAGED, MINB>)},

#define MOE_STEP_EXT_TABLE(NAME, ARRAY)                      \
  const StepExtVariant* NAME(int* n) {                       \
    *n = int(sizeof(ARRAY) / sizeof(ARRAY[0]));              \
    return ARRAY;                                            \
  }

#define MOE_VARIANT_TABLE(NAME, ARRAY)                       \
  const RouterVariant* NAME(int* n) {                        \
    *n = int(sizeof(ARRAY) / sizeof(ARRAY[0]));              \
    return ARRAY;                                            \
  }
