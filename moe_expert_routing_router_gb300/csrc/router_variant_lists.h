// The row layouts compiled for each element type and load path, as X-macro
// lists: the plain kernels' tables and the extended step's use the same lists.
// X(DT, LPR, VW, NV, NR, STAGED, MINB); the E each row covers is LPR * VW * NV.
#pragma once

// bf16 logits, rows streamed through the shared-memory ring (E % 8 == 0)
#define MOE_BF16_STAGED_LIST(X)                                                   \
  X(Bf16, 8, 1, 1, 2, true, 1)     /* E = 8 */                                    \
  X(Bf16, 8, 2, 1, 2, true, 1)     /* E = 16 */                                   \
  X(Bf16, 8, 4, 1, 2, true, 1)     /* E <= 32 */                                  \
  X(Bf16, 8, 8, 1, 2, true, 1)     /* E <= 64 */                                  \
  X(Bf16, 16, 8, 1, 2, true, 1)    /* E <= 128 */                                 \
  X(Bf16, 32, 8, 1, 2, true, 1)    /* E <= 256 (two rows per warp: 1.5 % faster at E = 256) */ \
  X(Bf16, 32, 4, 3, 1, true, 1)    /* E <= 384 */                                 \
  X(Bf16, 32, 8, 2, 1, true, 1)    /* E <= 512 */                                 \
  X(Bf16, 32, 8, 3, 1, true, 1)    /* E <= 768 */                                 \
  X(Bf16, 32, 8, 4, 1, true, 1)    /* E <= 1024 */

// bf16 logits of any E, read from global memory one element per load
#define MOE_BF16_DIRECT_LIST(X)                                                   \
  X(Bf16, 8, 1, 1, 1, false, 1)    /* E <= 8 */                                   \
  X(Bf16, 32, 1, 1, 1, false, 1)   /* E <= 32 */                                  \
  X(Bf16, 32, 1, 2, 1, false, 1)                                                  \
  X(Bf16, 32, 1, 4, 1, false, 1)                                                  \
  X(Bf16, 32, 1, 8, 1, false, 1)                                                  \
  X(Bf16, 32, 1, 16, 1, false, 1)                                                 \
  X(Bf16, 32, 1, 32, 1, false, 1)  /* E <= 1024 */

// fp32 logits, rows streamed through the shared-memory ring (E % 4 == 0)
#define MOE_FP32_STAGED_LIST(X)                                                   \
  X(Fp32, 8, 1, 1, 2, true, 1)     /* E <= 8 */                                   \
  X(Fp32, 8, 4, 1, 2, true, 1)     /* E <= 32 */                                  \
  X(Fp32, 8, 4, 2, 2, true, 1)     /* E <= 64 */                                  \
  X(Fp32, 16, 4, 2, 2, true, 1)    /* E <= 128 */                                 \
  X(Fp32, 32, 4, 2, 2, true, 1)    /* E <= 256 */                                 \
  X(Fp32, 32, 4, 3, 1, true, 1)    /* E <= 384 */                                 \
  X(Fp32, 32, 4, 4, 1, true, 1)    /* E <= 512 */                                 \
  X(Fp32, 32, 4, 8, 1, true, 1)    /* E <= 1024 */

// fp32 logits of any E, read from global memory one element per load
#define MOE_FP32_DIRECT_LIST(X)                                                   \
  X(Fp32, 8, 1, 1, 1, false, 1)    /* E <= 8 */                                   \
  X(Fp32, 32, 1, 1, 1, false, 1)   /* E <= 32 */                                  \
  X(Fp32, 32, 1, 2, 1, false, 1)                                                  \
  X(Fp32, 32, 1, 4, 1, false, 1)                                                  \
  X(Fp32, 32, 1, 8, 1, false, 1)                                                  \
  X(Fp32, 32, 1, 16, 1, false, 1)                                                 \
  X(Fp32, 32, 1, 32, 1, false, 1)  /* E <= 1024 */
