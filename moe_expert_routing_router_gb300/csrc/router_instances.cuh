// Explicit instantiation helpers for the router kernel variants.
#pragma once

#include "router_kernels.cuh"
#include "router_table.h"

#define MOE_ROUTER_VARIANT(DT, LPR, VW, NV, NR, STAGED, MINB)                                                       \
  {LPR, VW, NV, NR, STAGED, MINB,                                                                                    \
   reinterpret_cast<const void*>(&::moe::router_persistent_kernel<DT, LPR, VW, NV, NR, ::moe::kModeFwd, STAGED, MINB>), \
   reinterpret_cast<const void*>(&::moe::router_persistent_kernel<DT, LPR, VW, NV, NR, ::moe::kModeStep, STAGED, MINB>), \
   reinterpret_cast<const void*>(&::moe::router_bwd_kernel<DT, LPR, VW, NV>)}

#define MOE_VARIANT_TABLE(NAME, ARRAY)                       \
  const RouterVariant* NAME(int* n) {                        \
    *n = int(sizeof(ARRAY) / sizeof(ARRAY[0]));              \
    return ARRAY;                                            \
  }
