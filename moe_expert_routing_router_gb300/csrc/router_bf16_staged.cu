// bf16 logits, rows streamed through the shared-memory ring (E % 8 == 0).
#include "router_instances.cuh"
#include "router_variant_lists.h"

namespace moe {

static const RouterVariant kVariants[] = {MOE_BF16_STAGED_LIST(MOE_ROUTER_VARIANT_ITEM)};

MOE_VARIANT_TABLE(router_variants_bf16_staged, kVariants)

}  // namespace moe
