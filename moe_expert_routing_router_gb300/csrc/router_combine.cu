// The shard-combine kernel of the data-parallel statistics and the cross-rank
// exclusive scan of the expert counts (both declared in router_ext.cuh).
#include "router_ext.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) router_combine_kernel(const CombineParams p) {
  __shared__ int s_cnt[1024];
  __shared__ double s_pe[1024];
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    long long c = 0;
    double ps = 0.0;
    for (int g = 0; g < p.G; ++g) {
      c += p.counts[(long long)g * p.E + e];
      ps += double(p.P[(long long)g * p.E + e]) * p.T_shard[g];
    }
    s_cnt[e] = int(c);
    s_pe[e] = p.masked_p ? ps * double(p.k) : ps;     // the sum of p (over the picks when masked)
  }
  __syncthreads();
  FwdExParams q;
  memset(&q, 0, sizeof(q));
  q.T = p.T;
  q.E = p.E;
  q.k = p.k;
  q.masked_p = p.masked_p;
  q.alpha = p.alpha;
  q.n_ranks = p.n_ranks;
  q.counts = p.counts_out;
  q.f = p.f;
  q.P = p.P_out;
  q.scalars = p.scalars;
  q.rank_load = p.rank_load;
  ext_outputs(q, s_cnt, s_pe);
}

// base[e] = sum over ranks g < rank of counts[g][e]: every expert's exclusive
// scan across the data-parallel ranks, summed in 64 bits and clamped to int32.
__global__ void __launch_bounds__(256) shard_capacity_base_kernel(const int32_t* counts, int G, int E, int rank,
                                                                  int32_t* base) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    long long c = 0;
    for (int g = 0; g < rank && g < G; ++g) c += counts[(long long)g * E + e];
    base[e] = int32_t(c < 0x7fffffffLL ? c : 0x7fffffffLL);
  }
}

}  // namespace

cudaError_t launch_shard_capacity_base(const int32_t* counts, int G, int E, int rank, int32_t* base,
                                       cudaStream_t stream) {
  shard_capacity_base_kernel<<<(E + 255) / 256, 256, 0, stream>>>(counts, G, E, rank, base);
  return cudaGetLastError();
}

cudaError_t launch_router_combine(const CombineParams& p, cudaStream_t stream) {
  router_combine_kernel<<<1, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
