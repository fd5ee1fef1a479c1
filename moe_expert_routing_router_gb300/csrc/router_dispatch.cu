// The dispatch-only persistent kernel (the row layout parameters are unused).
#include "router_instances.cuh"

namespace moe {

const void* dispatch_kernel() {
  return reinterpret_cast<const void*>(
      &router_persistent_kernel<Bf16, 32, 1, 1, 1, kModeDispatch, false, kDispatchMinBlocks>);
}

}  // namespace moe
