// Launcher of the batched EPLB planner (expert replication and balanced packing).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kEplbMaxPhys = 4096;     // physical expert slots per problem
constexpr int kEplbMaxGpus = 256;      // GPUs (packing bins) per problem

struct EplbParams {
  const int32_t* loads;   // [B, E] token counts per expert (>= 0)
  int B, E;
  int num_phys, num_gpus, num_nodes, num_groups;
  int hier;               // hierarchical policy (groups onto nodes, then within each node)
  int32_t* phy2log;       // [B, num_phys]: logical expert of each physical slot, GPU-major
  int32_t* log_count;     // [B, E]: copies of each logical expert
  float* gpu_load;        // [B, num_gpus]: load of each GPU (sum of its copies' w / c)
};

// Dynamic shared memory of one CTA (one problem) for these sizes.
size_t eplb_smem_bytes(int E, int num_phys, int num_groups);
cudaError_t launch_eplb_plan(const EplbParams& p, cudaStream_t stream);

}  // namespace moe
