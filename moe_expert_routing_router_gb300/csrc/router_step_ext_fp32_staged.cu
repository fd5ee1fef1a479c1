// The extended step kernels: fp32 logits, rows streamed through the shared-memory ring (E % 4 == 0).
#include "router_instances.cuh"
#include "router_variant_lists.h"

namespace moe {

static const StepExtVariant kVariants[] = {MOE_FP32_STAGED_LIST(MOE_STEP_EXT_VARIANT_ITEM)};

MOE_STEP_EXT_TABLE(step_ext_fp32_staged, kVariants)

}  // namespace moe
