// bf16 logits, rows streamed through the shared-memory ring (E % 8 == 0).
#include "router_instances.cuh"

namespace moe {

static const RouterVariant kVariants[] = {
    MOE_ROUTER_VARIANT(Bf16, 8, 1, 1, 2, true, 1),     // E = 8
    MOE_ROUTER_VARIANT(Bf16, 8, 2, 1, 2, true, 1),     // E = 16
    MOE_ROUTER_VARIANT(Bf16, 8, 4, 1, 2, true, 1),     // E <= 32
    MOE_ROUTER_VARIANT(Bf16, 8, 8, 1, 2, true, 1),     // E <= 64
    MOE_ROUTER_VARIANT(Bf16, 16, 8, 1, 2, true, 1),    // E <= 128
    MOE_ROUTER_VARIANT(Bf16, 32, 8, 1, 2, true, 1),    // E <= 256 (two rows per warp: 1.5 % faster at E = 256)
    MOE_ROUTER_VARIANT(Bf16, 32, 4, 3, 1, true, 1),    // E <= 384
    MOE_ROUTER_VARIANT(Bf16, 32, 8, 2, 1, true, 1),    // E <= 512
    MOE_ROUTER_VARIANT(Bf16, 32, 8, 3, 1, true, 1),    // E <= 768
    MOE_ROUTER_VARIANT(Bf16, 32, 8, 4, 1, true, 1),    // E <= 1024
};

MOE_VARIANT_TABLE(router_variants_bf16_staged, kVariants)

}  // namespace moe
