// The extended step kernels: bf16 logits, rows streamed through the shared-memory ring (E % 8 == 0).
#include "router_instances.cuh"
#include "router_variant_lists.h"

namespace moe {

static const StepExtVariant kVariants[] = {MOE_BF16_STAGED_LIST(MOE_STEP_EXT_VARIANT_ITEM)};

MOE_STEP_EXT_TABLE(step_ext_bf16_staged, kVariants)

}  // namespace moe
