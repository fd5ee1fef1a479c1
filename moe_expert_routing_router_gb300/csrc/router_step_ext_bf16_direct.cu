// The extended step kernels: bf16 logits of any E, read from global memory one element per load.
#include "router_instances.cuh"
#include "router_variant_lists.h"

namespace moe {

static const StepExtVariant kVariants[] = {MOE_BF16_DIRECT_LIST(MOE_STEP_EXT_VARIANT_ITEM)};

MOE_STEP_EXT_TABLE(step_ext_bf16_direct, kVariants)

}  // namespace moe
