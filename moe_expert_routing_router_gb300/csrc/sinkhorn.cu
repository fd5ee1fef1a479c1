// TAOT Phase 1: the batched topology-aware Sinkhorn-Knopp flow plan.
//
// The topology cost takes three values (0 on the diagonal, 1 within a node,
// lambda across nodes), so the Gibbs kernel M = exp(-W/eps) is fixed by three
// numbers and (M x)_r needs only x_r, the sum S_n of x over rank r's node n
// and the total S:
//   (M x)_r = x_r + m_node (S_n - x_r) + m_cross (S - S_n)
//           = c_self x_r + c_node S_n + c_all S,
//   c_self = 1 - m_node,  c_node = m_node - m_cross,  c_all = m_cross.
// That is the dense product regrouped (the same value up to fp32 rounding) at
// O(R) per iteration instead of O(R^2).  M is symmetric, so M^T u is the same
// formula applied to u.
//
// One warp per microbatch: lane l holds ranks l and l + 32.  When
// ranks_per_node is a power of two up to 32, a node is an aligned group of
// lanes and the node sums and the total come from one butterfly (five shuffle
// levels, the two ranks interleaved); otherwise the node sums come from one
// pass over a shared-memory copy of x.  The plan diag(u) M diag(v) is written
// row by row, coalesced across the lanes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sinkhorn.h"

namespace moe {

constexpr int kSkWarps = 4;          // microbatches per CTA
constexpr int kSkRanks = 64;         // the largest supported rank count
constexpr float kDenFloor = 1e-30f;

__device__ __forceinline__ float sk_warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ float sk_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// y = M x for the warp's two ranks (node0 / node1: their node ids).
template <bool POW2>
__device__ __forceinline__ void sk_apply(const SinkhornParams& p, int lane, int nodes, int node0, int node1, float x0,
                                         float x1, float* xs, float* ns, float& y0, float& y1) {
  float n0, n1, total;
  if constexpr (POW2) {
    // One butterfly: after the levels below ranks_per_node each lane holds its
    // node's sum, after all five the sum over its half of the ranks.
    float t0 = x0, t1 = x1;
    n0 = x0;
    n1 = x1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      t0 += __shfl_xor_sync(0xffffffffu, t0, off);
      t1 += __shfl_xor_sync(0xffffffffu, t1, off);
      const bool in_node = off < p.ranks_per_node;
      n0 = in_node ? t0 : n0;
      n1 = in_node ? t1 : n1;
    }
    total = t0 + t1;
  } else {
    const int rpn = p.ranks_per_node;
    xs[lane] = x0;
    xs[lane + 32] = x1;
    total = sk_warp_sum(x0 + x1);
    __syncwarp();
    for (int n = lane; n < nodes; n += 32) {
      float s = 0.f;
      for (int j = 0; j < rpn; ++j) s += xs[n * rpn + j];
      ns[n] = s;
    }
    __syncwarp();
    n0 = ns[node0];
    n1 = ns[node1];
    __syncwarp();                     // xs and ns are rewritten by the next product
  }
  y0 = fmaf(p.c_self, x0, fmaf(p.c_node, n0, p.c_all * total));
  y1 = fmaf(p.c_self, x1, fmaf(p.c_node, n1, p.c_all * total));
}

template <bool POW2>
__global__ void __launch_bounds__(kSkWarps * 32) taot_sinkhorn_kernel(const SinkhornParams p) {
  __shared__ float sh_x[kSkWarps][kSkRanks];
  __shared__ float sh_n[kSkWarps][kSkRanks];
  __shared__ float sh_u[kSkWarps][kSkRanks];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kSkWarps + wid;
  if (b >= p.B) return;                                  // whole warps; no CTA-wide sync below
  const int R = p.R, rpn = p.ranks_per_node, nodes = R / rpn;
  const int node0 = lane / rpn, node1 = (lane + 32) / rpn;   // < kSkRanks
  const bool act0 = lane < R, act1 = lane + 32 < R;
  const float* ld = p.loads + (size_t)b * R;
  const float l0 = act0 ? ld[lane] : 0.f, l1 = act1 ? ld[lane + 32] : 0.f;
  const float mean = sk_warp_sum(l0 + l1) / float(R);
  const float o0 = act0 ? fmaxf(l0 - mean, 0.f) : 0.f, o1 = act1 ? fmaxf(l1 - mean, 0.f) : 0.f;
  const float d0 = act0 ? fmaxf(mean - l0, 0.f) : 0.f, d1 = act1 ? fmaxf(mean - l1, 0.f) : 0.f;
  const float sa = sk_warp_sum(o0 + o1), sb = sk_warp_sum(d0 + d1);
  float* plan = p.plan ? p.plan + (size_t)b * R * R : nullptr;
  float* uo = p.u + (size_t)b * R;
  float* vo = p.v + (size_t)b * R;

  if (!(sa > 0.f) || !(sb > 0.f)) {                      // nothing to move: empty plan
    if (act0) { uo[lane] = 0.f; vo[lane] = 0.f; }
    if (act1) { uo[lane + 32] = 0.f; vo[lane + 32] = 0.f; }
    if (plan)
      for (int i = lane; i < R * R; i += 32) plan[i] = 0.f;
    if (lane == 0) p.status[b] = 1;
    return;
  }
  const float a0 = o0 / sa, a1 = o1 / sa, b0 = d0 / sb, b1 = d1 / sb;
  float* xs = sh_x[wid];
  float* ns = sh_n[wid];
  float u0 = 0.f, u1 = 0.f, v0 = act0 ? 1.f : 0.f, v1 = act1 ? 1.f : 0.f;
  for (int it = 0; it < p.iters; ++it) {
    float y0, y1;
    sk_apply<POW2>(p, lane, nodes, node0, node1, v0, v1, xs, ns, y0, y1);
    u0 = act0 ? a0 * sk_rcp(fmaxf(y0, kDenFloor)) : 0.f;
    u1 = act1 ? a1 * sk_rcp(fmaxf(y1, kDenFloor)) : 0.f;
    sk_apply<POW2>(p, lane, nodes, node0, node1, u0, u1, xs, ns, y0, y1);
    v0 = act0 ? b0 * sk_rcp(fmaxf(y0, kDenFloor)) : 0.f;
    v1 = act1 ? b1 * sk_rcp(fmaxf(y1, kDenFloor)) : 0.f;
  }
  if (act0) { uo[lane] = u0; vo[lane] = v0; }
  if (act1) { uo[lane + 32] = u1; vo[lane + 32] = v1; }
  if (plan) {
    float* us = sh_u[wid];
    float* vs = xs;                    // the products are done: reuse the warp's x buffer for v
    us[lane] = u0;
    us[lane + 32] = u1;
    vs[lane] = v0;
    vs[lane + 32] = v1;
    __syncwarp();
    const int rpn = p.ranks_per_node;
    if (p.plan_vec4) {                 // R % 4 == 0 and a 16-byte aligned plan (checked on the host)
      // float4 stores: half-warp h writes row r + h, lane j its columns 4j .. 4j + 3.
      const int h = lane >> 4, j = lane & 15, c0 = 4 * j;
      const bool colok = c0 < R;
      float vc[4];
      int nc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        vc[i] = colok ? vs[c0 + i] : 0.f;
        nc[i] = (c0 + i) / rpn;
      }
      for (int r = h; r < R; r += 2) {
        const float ur = us[r];
        const int nr = r / rpn;
        float m[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) m[i] = r == c0 + i ? 1.f : (nr == nc[i] ? p.m_node : p.m_cross);
        if (colok)
          *reinterpret_cast<float4*>(plan + (size_t)r * R + c0) =
              make_float4(ur * m[0] * vc[0], ur * m[1] * vc[1], ur * m[2] * vc[2], ur * m[3] * vc[3]);
      }
    } else {
      for (int r = 0, nr = 0, left = rpn; r < R; ++r) {
        const float ur = us[r];
        float* row = plan + (size_t)r * R;
        const float m0 = r == lane ? 1.f : (nr == node0 ? p.m_node : p.m_cross);
        const float m1 = r == lane + 32 ? 1.f : (nr == node1 ? p.m_node : p.m_cross);
        if (act0) row[lane] = ur * m0 * v0;
        if (act1) row[lane + 32] = ur * m1 * v1;
        if (--left == 0) { ++nr; left = rpn; }
      }
    }
  }
  if (lane == 0) p.status[b] = 0;
}

cudaError_t launch_taot_sinkhorn(const SinkhornParams& p, cudaStream_t stream) {
  const int grid = (p.B + kSkWarps - 1) / kSkWarps;
  const int rpn = p.ranks_per_node;
  if (rpn <= 32 && (rpn & (rpn - 1)) == 0)
    taot_sinkhorn_kernel<true><<<grid, kSkWarps * 32, 0, stream>>>(p);
  else
    taot_sinkhorn_kernel<false><<<grid, kSkWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
