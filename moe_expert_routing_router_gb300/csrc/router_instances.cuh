// Explicit instantiation helpers for the router kernel variants.
#pragma once

#include "router_kernels.cuh"
#include "router_table.h"

#define MOE_ROUTER_VARIANT(DT, LPR, VW, NV)                                               \
  {LPR, VW, NV,                                                                          \
   reinterpret_cast<const void*>(&::moe::router_persistent_kernel<DT, LPR, VW, NV, ::moe::kModeFwd>), \
   reinterpret_cast<const void*>(&::moe::router_persistent_kernel<DT, LPR, VW, NV, ::moe::kModeStep>), \
   reinterpret_cast<const void*>(&::moe::router_bwd_kernel<DT, LPR, VW, NV>)}
