// fp32 logits of any E, read from global memory one element per load.
#include "router_instances.cuh"
#include "router_variant_lists.h"

namespace moe {

static const RouterVariant kVariants[] = {MOE_FP32_DIRECT_LIST(MOE_ROUTER_VARIANT_ITEM)};

MOE_VARIANT_TABLE(router_variants_fp32_direct, kVariants)

}  // namespace moe
