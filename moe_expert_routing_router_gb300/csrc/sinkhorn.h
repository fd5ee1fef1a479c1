// Launcher of the batched topology-aware Sinkhorn kernel.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

struct SinkhornParams {
  const float* loads;    // [B, R]
  int B, R, ranks_per_node, iters;
  float m_node;          // exp(-1 / eps): kernel value between two ranks of one node
  float m_cross;         // exp(-lambda / eps): kernel value across nodes
  float c_self;          // 1 - m_node
  float c_node;          // m_node - m_cross
  float c_all;           // m_cross
  float* u;              // [B, R]
  float* v;              // [B, R]
  float* plan;           // [B, R, R] or null
  int plan_vec4;         // 1: R % 4 == 0 and plan 16-byte aligned (rows written with float4 stores)
  int32_t* status;       // [B]
};

cudaError_t launch_taot_sinkhorn(const SinkhornParams& p, cudaStream_t stream);

}  // namespace moe
