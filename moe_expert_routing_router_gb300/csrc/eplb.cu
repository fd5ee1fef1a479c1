// Batched EPLB planner: expert replication and balanced packing onto GPUs, as
// the EPLB section (4.1.2) of the large-model load-balancing survey describes
// them ("企业官网建设流程全解析", cnvsn.com/news/335486):
//
//   replicate_experts  repeatedly adds a copy of the expert whose load per
//                      copy (weight / count) is largest, until the physical
//                      slot count is reached;
//   balanced_packing   takes the items heaviest first and puts each into the
//                      currently lightest bin that is not yet full (every bin
//                      takes the same number of items);
//   hierarchical       groups onto nodes by balanced_packing, then replication
//                      and packing onto the node's GPUs within each node (used
//                      when the node count divides the group count);
//   global             replication over all experts, packing onto all GPUs.
//
// One warp per problem, up to eight problems per CTA.  The replication compares w_a / c_a with w_b / c_b
// exactly (w_a * c_b against w_b * c_a in 64-bit integers), ties to the lower
// expert index.  The packing works in fp32: a copy weighs fp32(w) / fp32(c)
// (one rounding), a group fp32 of its integer sum, and a bin's total is the
// fp32 sum of its items in placement order; the sort is by weight descending,
// ties to the lower item index, and the lightest non-full bin wins, ties to
// the lower bin index.  Each warp runs its problem's two sequential greedy
// loops; the CTA shares the sorts (every item's rank counted against all others).
#include "eplb.h"

#include <float.h>

namespace moe {
namespace {

constexpr int kEplbThreads = 256;
constexpr int kEplbCountSort = 128;   // sets of up to this many items are sorted by counting

struct EplbSmem {
  int32_t* w;        // [E]  weights of the current sub-problem's experts (local order)
  int32_t* list;     // [E]  local expert -> global expert
  int32_t* cnt;      // [E]  copies per local expert
  int32_t* p2l;      // [num_phys] item -> local expert (item < n: first copy)
  float* x;          // [max(num_phys, num_groups)] item weights of a packing
  int32_t* order;    // [max(num_phys, num_groups), for the global policy rounded up to a power of two] sorted position -> item
  int32_t* gbin;     // [num_groups] node of each group
  int32_t* ginv;     // [num_groups] node-major: (node, position) -> group
  int order_cap;     // entries of order
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) / 16 * 16; }

__host__ __device__ inline size_t eplb_layout(int E, int num_phys, int num_groups, EplbSmem* s, char* base) {
  const int items = num_phys > num_groups ? num_phys : num_groups;
  // the global policy sorts all num_phys items at once, padded to a power of
  // two for the bitonic network; the hierarchical policy's sets are sorted by
  // counting (sort_items falls back to it wherever the padding is missing)
  int items_p2 = items;
  if (num_groups == 0 && items > kEplbCountSort) {
    items_p2 = 1;
    while (items_p2 < items) items_p2 <<= 1;
  }
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off += align16(bytes); return base ? base + o : nullptr; };
  char* w = take(4u * E);
  char* list = take(4u * E);
  char* cnt = take(4u * E);
  char* p2l = take(4u * num_phys);
  char* x = take(4u * items);
  char* order = take(4u * items_p2);
  char* gbin = take(4u * (num_groups > 0 ? num_groups : 1));
  char* ginv = take(4u * (num_groups > 0 ? num_groups : 1));
  if (s) {
    s->w = reinterpret_cast<int32_t*>(w);
    s->list = reinterpret_cast<int32_t*>(list);
    s->cnt = reinterpret_cast<int32_t*>(cnt);
    s->p2l = reinterpret_cast<int32_t*>(p2l);
    s->x = reinterpret_cast<float*>(x);
    s->order = reinterpret_cast<int32_t*>(order);
    s->gbin = reinterpret_cast<int32_t*>(gbin);
    s->ginv = reinterpret_cast<int32_t*>(ginv);
    s->order_cap = items_p2;
  }
  return off;
}

// w_a / c_a > w_b / c_b, or equal with a < b.
__device__ __forceinline__ bool heavier_per_copy(int32_t wa, int32_t ca, int a, int32_t wb, int32_t cb, int b) {
  const long long l = (long long)wa * cb, r = (long long)wb * ca;
  return l > r || (l == r && a < b);
}

// replicate_experts on the n experts in s.w: s.cnt and s.p2l for n_phys items
// (the calling warp alone).
__device__ void replicate_warp(const EplbSmem& s, int n, int n_phys) {
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < n; i += 32) {
    s.cnt[i] = 1;
    s.p2l[i] = i;
  }
  __syncwarp();
  for (int item = n; item < n_phys; ++item) {
    int best = -1;
    int32_t bw = 0, bc = 1;
    for (int i = lane; i < n; i += 32) {
      const int32_t wi = s.w[i], ci = s.cnt[i];
      if (best < 0 || heavier_per_copy(wi, ci, i, bw, bc, best)) {
        best = i;
        bw = wi;
        bc = ci;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const int ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int32_t ow = __shfl_xor_sync(0xffffffffu, bw, off), oc = __shfl_xor_sync(0xffffffffu, bc, off);
      if (ob >= 0 && (best < 0 || heavier_per_copy(ow, oc, ob, bw, bc, best))) {
        best = ob;
        bw = ow;
        bc = oc;
      }
    }
    if (lane == 0) {
      s.cnt[best] += 1;
      s.p2l[item] = best;
    }
    __syncwarp();
  }
}

// The CTA's problems share one shared-memory block each (`stride` bytes apart).
struct EplbCta {
  char* smem;
  size_t stride;
  int E, num_phys, num_groups;
  int n_active;                        // problems of this CTA (its first warps)
  __device__ EplbSmem at(int q) const {
    EplbSmem s;
    eplb_layout(E, num_phys, num_groups, &s, smem + size_t(q) * stride);
    return s;
  }
};

// Item a comes before item b in the packing order: the larger weight first,
// ties to the lower index; the padding (indices >= N) last.
__device__ __forceinline__ bool packs_before(const float* x, int N, int a, int b) {
  if (a >= N) return false;
  if (b >= N) return true;
  const float xa = x[a], xb = x[b];
  return xa > xb || (xa == xb && a < b);
}

// order[0..P) = the indices 0..N-1 in packing order, then the padding: a
// bitonic network by one warp (out of line, so that it does not weigh on the
// register allocation of the kernel's greedy loops).
__device__ __noinline__ void bitonic_order(const float* x, int32_t* order, int N, int P, int lane) {
  for (int i = lane; i < P; i += 32) order[i] = i;
  __syncwarp();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = lane; t < P / 2; t += 32) {
        const int i = 2 * t - (t & (stride - 1));            // the pair (i, i + stride)
        const int j = i + stride;
        const int a = order[i], b = order[j];
        const bool up = (i & size) == 0;                     // this block sorts in packing order
        if (up ? packs_before(x, N, b, a) : packs_before(x, N, a, b)) {
          order[i] = b;
          order[j] = a;
        }
      }
      __syncwarp();
    }
  }
}

// The packing order of every active problem's N items in s.x (weight
// descending, ties to the lower index).  Up to kEplbCountSort items, or where
// the order array has no room for the padding, each item counts the items
// that sort before it (all threads of the CTA, problem by problem); beyond,
// warp q sorts problem q's item indices, padded to a power of two, with a
// bitonic network in shared memory.  Called by all threads of the CTA.
__device__ void sort_items(const EplbCta& cta, int N) {
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int P = 1;
  while (P < N) P <<= 1;
  if (N <= kEplbCountSort || P > cta.at(0).order_cap) {
    for (int q = 0; q < cta.n_active; ++q) {
      const EplbSmem s = cta.at(q);
      for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const float xi = s.x[i];
        int r = 0;
        for (int j = 0; j < N; ++j) {
          const float xj = s.x[j];
          r += (xj > xi || (xj == xi && j < i)) ? 1 : 0;
        }
        s.order[r] = i;
      }
    }
  } else if (warp < cta.n_active) {
    bitonic_order(cta.at(warp).x, cta.at(warp).order, N, P, lane);
  }
  __syncthreads();
}

// balanced_packing of the N items (sorted in s.order) into G bins of N / G
// items, by the calling warp.  place(item, bin, position) is called in
// placement order; the bins' totals end in tot_out[bin] (when not null).
template <int kBinsPerLane, class Place>
__device__ void pack_warp_bpl(const EplbSmem& s, int N, int G, float* tot_out, Place place) {
  const int lane = threadIdx.x & 31;
  const int cap = N / G;
  float tot[kBinsPerLane];
  int fill[kBinsPerLane];
#pragma unroll
  for (int m = 0; m < kBinsPerLane; ++m) {
    tot[m] = 0.f;
    fill[m] = 0;
  }
  for (int q = 0; q < N; ++q) {
    const int item = s.order[q];
    // the lane's lightest open bin (its bins ascend with m: strict < keeps the lowest index)
    float bt = FLT_MAX;
    int bb = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < kBinsPerLane; ++m) {
      const int b = lane + 32 * m;
      if (b < G && fill[m] < cap && (bb == 0x7fffffff || tot[m] < bt)) {
        bt = tot[m];
        bb = b;
      }
    }
    // The warp's lightest open bin by two warp reductions: the smallest total
    // (totals are sums of non-negative weights, so their bit patterns order as
    // their values; a lane with no open bin offers the largest pattern), then
    // the lowest bin index holding it.
    const uint32_t img = bb == 0x7fffffff ? 0xffffffffu : __float_as_uint(bt);
    const uint32_t mt = __reduce_min_sync(0xffffffffu, img);
    bb = int(__reduce_min_sync(0xffffffffu, img == mt ? uint32_t(bb) : 0xffffffffu));
    if ((bb & 31) == lane) {
      const float xi = s.x[item];
#pragma unroll
      for (int m = 0; m < kBinsPerLane; ++m)
        if (m == (bb >> 5)) {
          place(item, bb, fill[m]);
          fill[m] += 1;
          tot[m] = __fadd_rn(tot[m], xi);
        }
    }
  }
  if (tot_out != nullptr) {
#pragma unroll
    for (int m = 0; m < kBinsPerLane; ++m)
      if (lane + 32 * m < G) tot_out[lane + 32 * m] = tot[m];
  }
  __syncwarp();
}

// Each lane holds ceil(G / 32) bins: 1, 2 or up to 8 (G <= 256).
template <class Place>
__device__ void pack_warp(const EplbSmem& s, int N, int G, float* tot_out, Place place) {
  if (G <= 32) pack_warp_bpl<1>(s, N, G, tot_out, place);
  else if (G <= 64) pack_warp_bpl<2>(s, N, G, tot_out, place);
  else pack_warp_bpl<kEplbMaxGpus / 32>(s, N, G, tot_out, place);
}

// Replication of each active problem's n experts (in s.w / s.list) onto n_phys
// slots, packed onto GPUs [gpu0, gpu0 + G) of the problem.  Called by the whole
// CTA; warp q works on problem `b` (active or not).
__device__ void solve(const EplbCta& cta, const EplbSmem& s, const EplbParams& p, int b, bool active, int n,
                      int n_phys, int G, int gpu0) {
  const int lane = threadIdx.x & 31;
  if (active) {
    replicate_warp(s, n, n_phys);
    for (int item = lane; item < n_phys; item += 32) {
      const int e = s.p2l[item];
      s.x[item] = __fdiv_rn(__int2float_rn(s.w[e]), __int2float_rn(s.cnt[e]));
    }
    for (int i = lane; i < n; i += 32) p.log_count[(long long)b * p.E + s.list[i]] = s.cnt[i];
  }
  sort_items(cta, n_phys);
  if (active) {
    const int S = p.num_phys / p.num_gpus;
    int32_t* out = p.phy2log + (long long)b * p.num_phys;
    pack_warp(s, n_phys, G, p.gpu_load + (long long)b * p.num_gpus + gpu0,
              [&](int item, int bin, int pos) { out[(gpu0 + bin) * S + pos] = s.list[s.p2l[item]]; });
  }
}

// One warp per problem, blockDim.x / 32 problems per CTA.
__global__ void __launch_bounds__(kEplbThreads) eplb_plan_kernel(const EplbParams p) {
  extern __shared__ __align__(16) char smem[];
  const int ppc = int(blockDim.x >> 5);
  const int wp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  EplbCta cta;
  cta.smem = smem;
  cta.stride = eplb_layout(p.E, p.num_phys, p.num_groups, nullptr, nullptr);
  cta.E = p.E;
  cta.num_phys = p.num_phys;
  cta.num_groups = p.num_groups;
  cta.n_active = min(ppc, p.B - int(blockIdx.x) * ppc);
  const int b = int(blockIdx.x) * ppc + wp;
  const bool active = wp < cta.n_active;
  const EplbSmem s = cta.at(wp);
  const int32_t* L = p.loads + (long long)(active ? b : 0) * p.E;
  if (!p.hier) {
    if (active) {
      for (int i = lane; i < p.E; i += 32) {
        s.w[i] = L[i];
        s.list[i] = i;
      }
      __syncwarp();
    }
    solve(cta, s, p, b, active, p.E, p.num_phys, p.num_gpus, 0);
    return;
  }
  // Groups onto nodes.
  const int gsize = p.E / p.num_groups;
  const int gpn_groups = p.num_groups / p.num_nodes;
  if (active) {
    for (int g = lane; g < p.num_groups; g += 32) {
      long long sum = 0;
      for (int j = 0; j < gsize; ++j) sum += L[g * gsize + j];
      s.x[g] = __ll2float_rn(sum);
    }
    __syncwarp();
  }
  sort_items(cta, p.num_groups);
  if (active)
    pack_warp(s, p.num_groups, p.num_nodes, nullptr, [&](int g, int node, int pos) {
      s.gbin[g] = node;
      s.ginv[node * gpn_groups + pos] = g;
    });
  // Within each node: its groups' experts in placement order.
  const int n = p.E / p.num_nodes;
  const int gpn = p.num_gpus / p.num_nodes;
  for (int node = 0; node < p.num_nodes; ++node) {
    if (active) {
      for (int j = lane; j < n; j += 32) {
        const int g = s.ginv[node * gpn_groups + j / gsize];
        const int e = g * gsize + j % gsize;
        s.list[j] = e;
        s.w[j] = L[e];
      }
      __syncwarp();
    }
    solve(cta, s, p, b, active, n, p.num_phys / p.num_nodes, gpn, node * gpn);
  }
}

}  // namespace

size_t eplb_smem_bytes(int E, int num_phys, int num_groups) { return eplb_layout(E, num_phys, num_groups, nullptr, nullptr); }

cudaError_t launch_eplb_plan(const EplbParams& p, cudaStream_t stream) {
  // As many problems per CTA (one warp each, at most 8) as leave room for two
  // CTAs in an SM's shared memory.
  constexpr size_t kSmemBudget = 100 * 1024;
  const size_t per = eplb_smem_bytes(p.E, p.num_phys, p.num_groups);
  int ppc = int(kSmemBudget / per);
  ppc = ppc < 1 ? 1 : (ppc > kEplbThreads / 32 ? kEplbThreads / 32 : ppc);
  const size_t smem = per * size_t(ppc);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(eplb_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  eplb_plan_kernel<<<(p.B + ppc - 1) / ppc, 32 * ppc, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
