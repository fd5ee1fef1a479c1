// TAOT Phase 1: the batched topology-aware Sinkhorn-Knopp flow plan.
//
// One CTA of 64 threads per microbatch; thread r owns rank r.  Supply, demand
// and the scaling vectors stay on chip for all iterations: thread r keeps row
// r of the Gibbs kernel M in registers, u and v live in shared memory.  The
// topology kernel is symmetric (W[r,s] = W[s,r]), so row r of M is also column
// r and serves both products M v and M^T u.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sinkhorn.h"

namespace moe {

constexpr int kSkThreads = 64;     // = the largest supported rank count
constexpr float kDenFloor = 1e-30f;

__device__ __forceinline__ float sum64(float x, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  return red[0] + red[1];
}

__device__ __forceinline__ float gibbs(int r, int s, int R, int rpn, float m_node, float m_cross) {
  if (r >= R || s >= R) return 0.f;
  if (r == s) return 1.f;
  return (r / rpn == s / rpn) ? m_node : m_cross;
}

__global__ void __launch_bounds__(kSkThreads) taot_sinkhorn_kernel(const SinkhornParams p) {
  __shared__ __align__(16) float sh_u[kSkThreads];
  __shared__ __align__(16) float sh_v[kSkThreads];
  __shared__ float red[2];
  const int b = blockIdx.x, r = threadIdx.x, R = p.R;
  const bool act = r < R;
  const float load = act ? p.loads[(size_t)b * R + r] : 0.f;
  const float mean = sum64(load, red) / float(R);
  const float over = act ? fmaxf(load - mean, 0.f) : 0.f;
  const float under = act ? fmaxf(mean - load, 0.f) : 0.f;
  const float sa = sum64(over, red);
  const float sb = sum64(under, red);
  float* plan = p.plan ? p.plan + (size_t)b * R * R : nullptr;

  if (!(sa > 0.f) || !(sb > 0.f)) {            // nothing to move: empty plan
    if (act) {
      p.u[(size_t)b * R + r] = 0.f;
      p.v[(size_t)b * R + r] = 0.f;
    }
    if (plan)
      for (int i = r; i < R * R; i += kSkThreads) plan[i] = 0.f;
    if (r == 0) p.status[b] = 1;
    return;
  }
  const float a = over / sa;
  const float bb = under / sb;

  float Mrow[kSkThreads];
#pragma unroll
  for (int s = 0; s < kSkThreads; ++s) Mrow[s] = gibbs(r, s, R, p.ranks_per_node, p.m_node, p.m_cross);

  sh_v[r] = act ? 1.f : 0.f;
  float u = 0.f, v = act ? 1.f : 0.f;
  for (int it = 0; it < p.iters; ++it) {
    __syncthreads();
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
    for (int s = 0; s < kSkThreads; s += 4) {
      const float4 vv = *reinterpret_cast<const float4*>(sh_v + s);
      acc0 = fmaf(Mrow[s], vv.x, acc0);
      acc1 = fmaf(Mrow[s + 1], vv.y, acc1);
      acc2 = fmaf(Mrow[s + 2], vv.z, acc2);
      acc3 = fmaf(Mrow[s + 3], vv.w, acc3);
    }
    u = act ? a / fmaxf((acc0 + acc1) + (acc2 + acc3), kDenFloor) : 0.f;
    sh_u[r] = u;
    __syncthreads();
    acc0 = acc1 = acc2 = acc3 = 0.f;
#pragma unroll
    for (int s = 0; s < kSkThreads; s += 4) {
      const float4 uu = *reinterpret_cast<const float4*>(sh_u + s);
      acc0 = fmaf(Mrow[s], uu.x, acc0);
      acc1 = fmaf(Mrow[s + 1], uu.y, acc1);
      acc2 = fmaf(Mrow[s + 2], uu.z, acc2);
      acc3 = fmaf(Mrow[s + 3], uu.w, acc3);
    }
    v = act ? bb / fmaxf((acc0 + acc1) + (acc2 + acc3), kDenFloor) : 0.f;
    sh_v[r] = v;
  }
  __syncthreads();
  sh_u[r] = u;
  __syncthreads();
  if (act) {
    p.u[(size_t)b * R + r] = u;
    p.v[(size_t)b * R + r] = v;
  }
  if (plan) {
    for (int i = r; i < R * R; i += kSkThreads) {
      const int rr = i / R, ss = i - rr * R;
      plan[i] = sh_u[rr] * gibbs(rr, ss, R, p.ranks_per_node, p.m_node, p.m_cross) * sh_v[ss];
    }
  }
  if (r == 0) p.status[b] = 0;
}

cudaError_t launch_taot_sinkhorn(const SinkhornParams& p, cudaStream_t stream) {
  taot_sinkhorn_kernel<<<p.B, kSkThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
