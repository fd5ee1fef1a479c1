// Launcher of the batched TAOT Phase 2 matching (hot experts onto cold ranks).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kMatchMaxRounds = 16;   // K, replicas per cold rank

struct MatchParams {
  const int32_t* expert_loads;   // [B, E]
  const float* plan;             // [B, R, R] Phase 1 flow, plan[h, c] from hot rank h to cold rank c
  int B, E, R, ranks_per_node, K;
  int32_t* slot_expert;          // [B, R, K] (-1: empty)
  int32_t* slot_tokens;          // [B, R, K]
  int32_t* rank_load;            // [B, R] after the moves
};

size_t taot_match_smem_bytes(int E, int R);
cudaError_t launch_taot_match(const MatchParams& p, cudaStream_t stream);

}  // namespace moe
