// The extended step kernels: fp32 logits of any E, read from global memory one element per load.
#include "router_instances.cuh"
#include "router_variant_lists.h"

namespace moe {

static const StepExtVariant kVariants[] = {MOE_FP32_DIRECT_LIST(MOE_STEP_EXT_VARIANT_ITEM)};

MOE_STEP_EXT_TABLE(step_ext_fp32_direct, kVariants)

}  // namespace moe
