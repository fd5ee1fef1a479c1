// fp32-logit router variants.  Vector variants need E % 4 == 0 and 16-byte
// aligned arrays; the VW == 1 variants take any E.
#include "router_instances.cuh"

namespace moe {

static const RouterVariant kFp32Variants[] = {
    MOE_ROUTER_VARIANT(Fp32, 8, 4, 1),     // E <= 32
    MOE_ROUTER_VARIANT(Fp32, 8, 4, 2),     // E <= 64
    MOE_ROUTER_VARIANT(Fp32, 16, 4, 2),    // E <= 128
    MOE_ROUTER_VARIANT(Fp32, 32, 4, 2),    // E <= 256
    MOE_ROUTER_VARIANT(Fp32, 32, 4, 3),    // E <= 384
    MOE_ROUTER_VARIANT(Fp32, 32, 4, 4),    // E <= 512
    MOE_ROUTER_VARIANT(Fp32, 32, 4, 8),    // E <= 1024
    MOE_ROUTER_VARIANT(Fp32, 8, 1, 1),     // any E <= 8
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 1),    // any E <= 32
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 2),
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 4),
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 8),
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 16),
    MOE_ROUTER_VARIANT(Fp32, 32, 1, 32),   // any E <= 1024
};

const RouterVariant* router_variants_fp32(int* n) {
  *n = int(sizeof(kFp32Variants) / sizeof(kFp32Variants[0]));
  return kFp32Variants;
}

}  // namespace moe
