// Batched TAOT Phase 2: column-first iterative matching of hot experts to cold
// ranks, as section 2 of the LoongForge TAOT article describes it ("MoE 训练端到端
// 加速 1.43 倍 ..."): rounds in which every cold rank picks its best hot expert on
// its own, conflicts over one expert are arbitrated, and a rank that lost picks
// again in the next round, until no cold rank finds a match; each cold rank
// hosts at most K replicas.
//
// The pair score is (tokens moved, same node, Phase 1 flow plan[h, c]), then the
// lower expert index; arbitration uses the same score, then the lower rank
// index.  A match (c, e) moves min(w_rem[e], floor(load[h] - mean),
// floor(mean - load[c])) tokens of expert e from its home rank h; the winners
// of a round commit in ascending rank order, each move taken again against the
// loads as they stand then.  Loads are compared with the mean exactly, as
// load * R against the total.
//
// One CTA per microbatch.  Each round first gathers the candidate experts
// (home rank hot, tokens left); a warp per cold rank scores them (lanes stride
// over the candidates, a shuffle tree picks the best); thread 0 arbitrates and
// commits, at most R moves per round.
#include "taot_match.h"

namespace moe {
namespace {

constexpr int kMatchThreads = 256;

struct Score {
  int x;        // tokens moved
  int same;     // 1: same node
  float flow;   // plan[h, c]
  int e;        // expert (ties: the lower wins)
};

__device__ __forceinline__ bool better(const Score& a, const Score& b) {   // a before b
  if (a.x != b.x) return a.x > b.x;
  if (a.same != b.same) return a.same > b.same;
  if (a.flow != b.flow) return a.flow > b.flow;
  return a.e < b.e;
}

struct MatchSmem {
  long long* load;     // [R]
  int32_t* w_rem;      // [E]
  uint32_t* used;      // [R][E / 32 rounded up]
  int32_t* n_slots;    // [R]
  int32_t* choice;     // [R] chosen expert or -1
  int32_t* ch_x;       // [R]
  int32_t* ch_same;    // [R]
  float* ch_flow;      // [R]
  int32_t* win;        // [E] winning rank of each expert this round, or -1
  int32_t* cand;       // [E] this round's candidates: experts on hot ranks with tokens left
  int32_t* n_cand;     // [1]
  int32_t* any;        // [1] the round had a choice (another round follows)
  long long* total;    // [1]
};

__host__ __device__ inline size_t a16(size_t x) { return (x + 15) / 16 * 16; }

__host__ __device__ inline size_t match_layout(int E, int R, MatchSmem* s, char* base) {
  const int words = (E + 31) / 32;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off += a16(bytes); return base ? base + o : nullptr; };
  char* load = take(8u * R);
  char* total = take(8u);
  char* w_rem = take(4u * E);
  char* used = take(4u * R * words);
  char* n_slots = take(4u * R);
  char* choice = take(4u * R);
  char* ch_x = take(4u * R);
  char* ch_same = take(4u * R);
  char* ch_flow = take(4u * R);
  char* win = take(4u * E);
  char* cand = take(4u * E);
  char* n_cand = take(4u);
  char* any = take(4u);
  if (s) {
    s->any = reinterpret_cast<int32_t*>(any);
    s->cand = reinterpret_cast<int32_t*>(cand);
    s->n_cand = reinterpret_cast<int32_t*>(n_cand);
    s->load = reinterpret_cast<long long*>(load);
    s->total = reinterpret_cast<long long*>(total);
    s->w_rem = reinterpret_cast<int32_t*>(w_rem);
    s->used = reinterpret_cast<uint32_t*>(used);
    s->n_slots = reinterpret_cast<int32_t*>(n_slots);
    s->choice = reinterpret_cast<int32_t*>(choice);
    s->ch_x = reinterpret_cast<int32_t*>(ch_x);
    s->ch_same = reinterpret_cast<int32_t*>(ch_same);
    s->ch_flow = reinterpret_cast<float*>(ch_flow);
    s->win = reinterpret_cast<int32_t*>(win);
  }
  return off;
}

// Tokens the match (c, e) would move now (0: none).
__device__ __forceinline__ int moved(const MatchSmem& s, int R, int per, int words, int c, int e) {
  const long long total = *s.total;
  const int h = e / per;
  const long long lh = s.load[h] * R, lc = s.load[c] * R;
  if (lh <= total || lc >= total || s.w_rem[e] <= 0 || ((s.used[c * words + (e >> 5)] >> (e & 31)) & 1u)) return 0;
  const long long excess = (lh - total) / R, spare = (total - lc) / R;
  long long x = s.w_rem[e];
  x = excess < x ? excess : x;
  x = spare < x ? spare : x;
  return x > 0 ? int(x) : 0;
}

__global__ void __launch_bounds__(kMatchThreads) taot_match_kernel(const MatchParams p) {
  extern __shared__ __align__(16) char smem[];
  MatchSmem s;
  match_layout(p.E, p.R, &s, smem);
  const int b = blockIdx.x, R = p.R, E = p.E, K = p.K, per = E / R, words = (E + 31) / 32;
  const int32_t* w = p.expert_loads + (long long)b * E;
  const float* plan = p.plan + (long long)b * R * R;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = kMatchThreads / 32;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    s.w_rem[e] = w[e];
    s.win[e] = -1;
  }
  for (int i = threadIdx.x; i < R * words; i += blockDim.x) s.used[i] = 0u;
  for (int r = threadIdx.x; r < R; r += blockDim.x) s.n_slots[r] = 0;
  int32_t* se = p.slot_expert + (long long)b * R * K;
  int32_t* st = p.slot_tokens + (long long)b * R * K;
  for (int i = threadIdx.x; i < R * K; i += blockDim.x) {
    se[i] = -1;
    st[i] = 0;
  }
  // rank loads: warp r sums its experts
  for (int r = warp; r < R; r += nwarps) {
    long long v = 0;
    for (int j = lane; j < per; j += 32) v += w[r * per + j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) s.load[r] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long t = 0;
    for (int r = 0; r < R; ++r) t += s.load[r];
    *s.total = t;
  }
  __syncthreads();
  // Rounds repeat while some cold rank still finds a positive match.  A round
  // with a choice commits at least its lowest-ranked winner (no earlier move of
  // the round changed its numbers), and a rank holds at most K replicas, so
  // there are at most R * K + 1 rounds.
  for (int round = 0; round <= R * K; ++round) {
    // This round's candidates: experts whose home rank is hot and that still
    // have tokens at home (in any order: the score breaks ties by index).
    if (threadIdx.x == 0) *s.n_cand = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
      if (s.load[e / per] * R > *s.total && s.w_rem[e] > 0) s.cand[atomicAdd(s.n_cand, 1)] = e;
    __syncthreads();
    const int n_cand = *s.n_cand;
    // Every cold rank with a free slot picks its best expert.
    for (int c = warp; c < R; c += nwarps) {
      Score best = {0, 0, 0.f, 0x7fffffff};
      if (s.n_slots[c] < K && s.load[c] * R < *s.total) {
        for (int q = lane; q < n_cand; q += 32) {
          const int e = s.cand[q];
          const int x = moved(s, R, per, words, c, e);
          if (x <= 0) continue;
          const int h = e / per;
          const Score sc = {x, (h / p.ranks_per_node) == (c / p.ranks_per_node) ? 1 : 0, plan[h * R + c], e};
          if (best.x == 0 || better(sc, best)) best = sc;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        Score o;
        o.x = __shfl_xor_sync(0xffffffffu, best.x, off);
        o.same = __shfl_xor_sync(0xffffffffu, best.same, off);
        o.flow = __shfl_xor_sync(0xffffffffu, best.flow, off);
        o.e = __shfl_xor_sync(0xffffffffu, best.e, off);
        if (o.x > 0 && (best.x == 0 || better(o, best))) best = o;
      }
      if (lane == 0) {
        s.choice[c] = best.x > 0 ? best.e : -1;
        s.ch_x[c] = best.x;
        s.ch_same[c] = best.same;
        s.ch_flow[c] = best.flow;
      }
    }
    __syncthreads();
    // Arbitration, then the winners' moves in ascending rank order.
    if (threadIdx.x == 0) {
      for (int c = 0; c < R; ++c) {
        const int e = s.choice[c];
        if (e < 0) continue;
        const int o = s.win[e];
        if (o < 0) {
          s.win[e] = c;
        } else {
          const Score a = {s.ch_x[c], s.ch_same[c], s.ch_flow[c], 0}, q = {s.ch_x[o], s.ch_same[o], s.ch_flow[o], 0};
          if (better(a, q)) s.win[e] = c;            // equal scores keep the lower rank
        }
      }
      for (int c = 0; c < R; ++c) {
        const int e = s.choice[c];
        if (e < 0 || s.win[e] != c) continue;
        const int x = moved(s, R, per, words, c, e);
        if (x > 0) {
          const int h = e / per;
          s.load[h] -= x;
          s.load[c] += x;
          s.w_rem[e] -= x;
          s.used[c * words + (e >> 5)] |= 1u << (e & 31);
          se[c * K + s.n_slots[c]] = e;
          st[c * K + s.n_slots[c]] = x;
          s.n_slots[c] += 1;
        }
      }
      int chosen = 0;
      for (int c = 0; c < R; ++c)
        if (s.choice[c] >= 0) {
          s.win[s.choice[c]] = -1;
          ++chosen;
        }
      *s.any = chosen;
    }
    __syncthreads();
    if (*s.any == 0) break;                   // written before the barrier, rewritten only after the next two
  }
  for (int r = threadIdx.x; r < R; r += blockDim.x) p.rank_load[(long long)b * R + r] = int32_t(s.load[r]);
}

}  // namespace

size_t taot_match_smem_bytes(int E, int R) { return match_layout(E, R, nullptr, nullptr); }

cudaError_t launch_taot_match(const MatchParams& p, cudaStream_t stream) {
  const size_t smem = taot_match_smem_bytes(p.E, p.R);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(taot_match_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  taot_match_kernel<<<p.B, kMatchThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
