// fp32 logits, rows streamed through the shared-memory ring (E % 4 == 0).
#include "router_instances.cuh"
#include "router_variant_lists.h"

namespace moe {

static const RouterVariant kVariants[] = {MOE_FP32_STAGED_LIST(MOE_ROUTER_VARIANT_ITEM)};

MOE_VARIANT_TABLE(router_variants_fp32_staged, kVariants)

}  // namespace moe
