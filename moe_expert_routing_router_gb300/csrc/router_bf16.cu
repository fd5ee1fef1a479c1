// bf16-logit router variants.  Vector variants need E % VW == 0 and 16-byte
// aligned arrays; the VW == 1 variants take any E.
#include "router_instances.cuh"

namespace moe {

static const RouterVariant kBf16Variants[] = {
    MOE_ROUTER_VARIANT(Bf16, 8, 2, 1),     // E <= 16
    MOE_ROUTER_VARIANT(Bf16, 8, 4, 1),     // E <= 32
    MOE_ROUTER_VARIANT(Bf16, 8, 8, 1),     // E <= 64
    MOE_ROUTER_VARIANT(Bf16, 16, 8, 1),    // E <= 128
    MOE_ROUTER_VARIANT(Bf16, 32, 8, 1),    // E <= 256
    MOE_ROUTER_VARIANT(Bf16, 32, 4, 3),    // E <= 384
    MOE_ROUTER_VARIANT(Bf16, 32, 8, 2),    // E <= 512
    MOE_ROUTER_VARIANT(Bf16, 32, 8, 3),    // E <= 768
    MOE_ROUTER_VARIANT(Bf16, 32, 8, 4),    // E <= 1024
    MOE_ROUTER_VARIANT(Bf16, 8, 1, 1),     // any E <= 8
    MOE_ROUTER_VARIANT(Bf16, 32, 1, 1),    // any E <= 32
    MOE_ROUTER_VARIANT(Bf16, 32, 1, 2),
    MOE_ROUTER_VARIANT(Bf16, 32, 1, 4),
    MOE_ROUTER_VARIANT(Bf16, 32, 1, 8),
    MOE_ROUTER_VARIANT(Bf16, 32, 1, 16),
    MOE_ROUTER_VARIANT(Bf16, 32, 1, 32),   // any E <= 1024
};

const RouterVariant* router_variants_bf16(int* n) {
  *n = int(sizeof(kBf16Variants) / sizeof(kBf16Variants[0]));
  return kBf16Variants;
}

}  // namespace moe
