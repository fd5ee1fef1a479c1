// fp32 logits of any E, read from global memory one element per load.
#include "router_instances.cuh"

namespace moe {

static const RouterVariant kVariants[] = {
    MOE_ROUTER_VARIANT(Fp32, 8, 1, 1, 1, false, 1),    // E <= 8
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 1, 1, false, 1),   // E <= 32
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 2, 1, false, 1),
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 4, 1, false, 1),
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 8, 1, false, 1),
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 16, 1, false, 1),
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 32, 1, false, 1),  // E <= 1024
};

MOE_VARIANT_TABLE(router_variants_fp32_direct, kVariants)

}  // namespace moe
