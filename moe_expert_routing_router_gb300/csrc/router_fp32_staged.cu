// fp32 logits, rows streamed through the shared-memory ring (E % 4 == 0).
#include "router_instances.cuh"

namespace moe {

static const RouterVariant kVariants[] = {
    MOE_ROUTER_VARIANT(Fp32, 8, 1, 1, 2, true, 1),     // E <= 8
    MOE_ROUTER_VARIANT(Fp32, 8, 4, 1, 2, true, 1),     // E <= 32
    MOE_ROUTER_VARIANT(Fp32, 8, 4, 2, 2, true, 1),     // E <= 64
    MOE_ROUTER_VARIANT(Fp32, 16, 4, 2, 2, true, 1),    // E <= 128
    MOE_ROUTER_VARIANT(Fp32, 32, 4, 2, 2, true, 1),    // E <= 256
    MOE_ROUTER_VARIANT(Fp32, 32, 4, 3, 1, true, 1),    // E <= 384
    MOE_ROUTER_VARIANT(Fp32, 32, 4, 4, 1, true, 1),    // E <= 512
    MOE_ROUTER_VARIANT(Fp32, 32, 4, 8, 1, true, 1),    // E <= 1024
};

MOE_VARIANT_TABLE(router_variants_fp32_staged, kVariants)

}  // namespace moe
