// bf16 instances of the full backward.
#include "router_ext.cuh"
#include "router_table.h"

#define MOE_EXT_VARIANT(DT, LPR, VW, NV, VEC)                                         \
  {LPR, VW, NV, VEC, reinterpret_cast<const void*>(&::moe::router_bwd_full_kernel<DT, LPR, VW, NV>)}

namespace moe {

static const ExtVariant kExtVariants[] = {
    // rows of a multiple of 16 bytes, 16-byte aligned
    MOE_EXT_VARIANT(Bf16, 8, 1, 1, 1),      // E = 8
    MOE_EXT_VARIANT(Bf16, 8, 2, 1, 1),      // E = 16
    MOE_EXT_VARIANT(Bf16, 8, 4, 1, 1),      // E <= 32
    MOE_EXT_VARIANT(Bf16, 8, 8, 1, 1),      // E <= 64
    MOE_EXT_VARIANT(Bf16, 16, 8, 1, 1),     // E <= 128
    MOE_EXT_VARIANT(Bf16, 32, 8, 1, 1),     // E <= 256
    MOE_EXT_VARIANT(Bf16, 32, 4, 3, 1),     // E <= 384
    MOE_EXT_VARIANT(Bf16, 32, 8, 2, 1),     // E <= 512
    MOE_EXT_VARIANT(Bf16, 32, 8, 4, 1),     // E <= 1024
    // any E and alignment, one element per load
    MOE_EXT_VARIANT(Bf16, 8, 1, 1, 0),      // E <= 8
    MOE_EXT_VARIANT(Bf16, 32, 1, 1, 0),     // E <= 32
    MOE_EXT_VARIANT(Bf16, 32, 1, 2, 0),
    MOE_EXT_VARIANT(Bf16, 32, 1, 4, 0),
    MOE_EXT_VARIANT(Bf16, 32, 1, 8, 0),
    MOE_EXT_VARIANT(Bf16, 32, 1, 16, 0),
    MOE_EXT_VARIANT(Bf16, 32, 1, 32, 0),    // E <= 1024
};

const ExtVariant* ext_variants_bf16(int* n) {
  *n = int(sizeof(kExtVariants) / sizeof(kExtVariants[0]));
  return kExtVariants;
}

}  // namespace moe
