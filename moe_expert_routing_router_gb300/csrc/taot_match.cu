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
// over the candidates, a shuffle tree picks the best).  The arbitration is two
// shared-memory atomic maxima per expert over its choosers' keys, (tokens,
// same node) and then (flow, inverted rank), so the best chooser and, among
// equal ones, the lowest rank wins.  The winners' moves are committed in
// ascending rank order within each hot home rank (the only quantity two
// winners of a round share is the load of the hot rank they both draw on) and
// in parallel across home ranks.  floor((load * R - total) / R) is
// load - ceil(total / R) and floor((total - load * R) / R) is
// floor(total / R) - load, so no division is left in the scoring.
#include "taot_match.h"

namespace moe {
namespace {

constexpr int kMatchThreads = 256;

struct MatchSmem {
  long long* load;     // [R]
  int32_t* w_rem;      // [E]
  uint32_t* used;      // [R][E / 32 rounded up]
  int32_t* n_slots;    // [R]
  int32_t* choice;     // [R] chosen expert or -1
  uint32_t* key1;      // [R] the choice's (tokens << 1) | same node
  unsigned long long* key2;   // [R] the choice's (flow image << 6) | (63 - rank)
  uint32_t* win1;      // [E] best key1 among the expert's choosers this round (0: none)
  unsigned long long* win2;   // [E] best key2 among the choosers with the best key1
  unsigned long long* hmask;  // [R] this round's winners drawing on hot home rank h, one bit per rank
  int32_t* cand;       // [E] this round's candidates: experts on hot ranks with tokens left
  int32_t* give;       // [E] per candidate: min(tokens left at home, floor(home load - mean))
  int32_t* hnode;      // [E] node of each expert's home rank
  float* plan;         // [R][R] this microbatch's Phase 1 flow
  int32_t* n_cand;     // [1]
  int32_t* any;        // [1] the round had a choice (another round follows)
  int32_t* steps;      // [1] the most winners on one home rank this round
  long long* total;    // [1]
};

__host__ __device__ inline size_t a16(size_t x) { return (x + 15) / 16 * 16; }

__host__ __device__ inline size_t match_layout(int E, int R, MatchSmem* s, char* base) {
  const int words = (E + 31) / 32;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off += a16(bytes); return base ? base + o : nullptr; };
  char* load = take(8u * R);
  char* total = take(8u);
  char* key2 = take(8u * R);
  char* win2 = take(8u * E);
  char* hmask = take(8u * R);
  char* w_rem = take(4u * E);
  char* used = take(4u * R * words);
  char* n_slots = take(4u * R);
  char* choice = take(4u * R);
  char* key1 = take(4u * R);
  char* win1 = take(4u * E);
  char* cand = take(4u * E);
  char* give = take(4u * E);
  char* hnode = take(4u * E);
  char* plan = take(4u * R * R);
  char* n_cand = take(4u);
  char* any = take(4u);
  char* steps = take(4u);
  if (s) {
    s->any = reinterpret_cast<int32_t*>(any);
    s->steps = reinterpret_cast<int32_t*>(steps);
    s->cand = reinterpret_cast<int32_t*>(cand);
    s->give = reinterpret_cast<int32_t*>(give);
    s->hnode = reinterpret_cast<int32_t*>(hnode);
    s->plan = reinterpret_cast<float*>(plan);
    s->n_cand = reinterpret_cast<int32_t*>(n_cand);
    s->load = reinterpret_cast<long long*>(load);
    s->total = reinterpret_cast<long long*>(total);
    s->w_rem = reinterpret_cast<int32_t*>(w_rem);
    s->used = reinterpret_cast<uint32_t*>(used);
    s->n_slots = reinterpret_cast<int32_t*>(n_slots);
    s->choice = reinterpret_cast<int32_t*>(choice);
    s->key1 = reinterpret_cast<uint32_t*>(key1);
    s->key2 = reinterpret_cast<unsigned long long*>(key2);
    s->win1 = reinterpret_cast<uint32_t*>(win1);
    s->win2 = reinterpret_cast<unsigned long long*>(win2);
    s->hmask = reinterpret_cast<unsigned long long*>(hmask);
  }
  return off;
}

// Tokens the match (c, e) would move now (0: none).  fl = floor(total / R),
// cl = ceil(total / R).
__device__ __forceinline__ int moved(const MatchSmem& s, int R, int per, int words, long long total, long long fl,
                                     long long cl, int c, int e) {
  const int h = e / per;
  const long long Lh = s.load[h], Lc = s.load[c];
  if (Lh * R <= total || Lc * R >= total || s.w_rem[e] <= 0 || ((s.used[c * words + (e >> 5)] >> (e & 31)) & 1u)) return 0;
  long long x = s.w_rem[e];
  x = Lh - cl < x ? Lh - cl : x;                 // floor(load_h - mean)
  x = fl - Lc < x ? fl - Lc : x;                 // floor(mean - load_c)
  return x > 0 ? int(x) : 0;
}

// Larger flow, larger image (-0 folded into +0 first).
__device__ __forceinline__ uint32_t flow_image(float f) {
  const uint32_t b = __float_as_uint(__fadd_rn(f, 0.f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kMatchThreads) taot_match_kernel(const MatchParams p) {
  extern __shared__ __align__(16) char smem[];
  MatchSmem s;
  match_layout(p.E, p.R, &s, smem);
  const int b = blockIdx.x, R = p.R, E = p.E, K = p.K, per = E / R, words = (E + 31) / 32;
  const int32_t* w = p.expert_loads + (long long)b * E;
  const float* plan = p.plan + (long long)b * R * R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = kMatchThreads / 32;
  for (int e = tid; e < E; e += blockDim.x) {
    s.w_rem[e] = w[e];
    s.win1[e] = 0u;
    s.win2[e] = 0ull;
    s.hnode[e] = (e / per) / p.ranks_per_node;
  }
  for (int i = tid; i < R * R; i += blockDim.x) s.plan[i] = plan[i];
  for (int i = tid; i < R * words; i += blockDim.x) s.used[i] = 0u;
  for (int r = tid; r < R; r += blockDim.x) {
    s.n_slots[r] = 0;
    s.hmask[r] = 0ull;
  }
  int32_t* se = p.slot_expert + (long long)b * R * K;
  int32_t* st = p.slot_tokens + (long long)b * R * K;
  for (int i = tid; i < R * K; i += blockDim.x) {
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
  if (tid == 0) {
    long long t = 0;
    for (int r = 0; r < R; ++r) t += s.load[r];
    *s.total = t;
  }
  __syncthreads();
  const long long total = *s.total;
  const long long fl = total >= 0 ? total / R : -((-total + R - 1) / R);
  const long long cl = total >= 0 ? (total + R - 1) / R : -((-total) / R);
  // Rounds repeat while some cold rank still finds a positive match.  A round
  // with a choice commits at least its lowest-ranked winner (no earlier move of
  // the round changed its numbers), and a rank holds at most K replicas, so
  // there are at most R * K + 1 rounds.
  for (int round = 0; round <= R * K; ++round) {
    // This round's candidates: experts whose home rank is hot and that still
    // have tokens at home (in any order: the score breaks ties by index).
    if (tid == 0) {
      *s.n_cand = 0;
      *s.any = 0;
      *s.steps = 0;
    }
    __syncthreads();
    for (int e0 = warp * 32; e0 < E; e0 += kMatchThreads) {   // whole warps: the ballot needs every lane
      const int e = e0 + lane;
      long long g = 0;
      if (e < E) {
        const long long Lh = s.load[e / per];
        if (Lh * R > total && s.w_rem[e] > 0) g = Lh - cl < s.w_rem[e] ? Lh - cl : s.w_rem[e];
      }
      const unsigned m = __ballot_sync(0xffffffffu, g > 0);
      int base = 0;
      if (lane == 0 && m != 0u) base = atomicAdd(s.n_cand, __popc(m));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (g > 0) {
        const int q = base + __popc(m & ((1u << lane) - 1u));
        s.cand[q] = e;
        s.give[q] = int(g);
      }
    }
    __syncthreads();
    const int n_cand = *s.n_cand;
    // Every cold rank with a free slot picks its best expert: the largest
    // (tokens << 1 | same node), then the largest flow, then the lowest expert:
    // each lane keeps its best in that order over its share of the candidates,
    // and three warp reductions settle the warp's.  A match moves
    // min(give, floor(mean - load_c)).
    for (int c = warp; c < R; c += nwarps) {
      uint32_t k1 = 0u, fimg = 0u;
      int be = 0x7fffffff;
      const long long Lc = s.load[c];
      if (s.n_slots[c] < K && Lc * R < total) {
        const long long spare = fl - Lc;
        const int node_c = c / p.ranks_per_node;
        for (int q = lane; q < n_cand; q += 32) {
          const int e = s.cand[q];
          if ((s.used[c * words + (e >> 5)] >> (e & 31)) & 1u) continue;
          const long long x = s.give[q] < spare ? s.give[q] : spare;
          if (x <= 0) continue;
          const uint32_t k = (uint32_t(x) << 1) | uint32_t(s.hnode[e] == node_c ? 1 : 0);
          if (k < k1) continue;
          const uint32_t fi = flow_image(s.plan[(e / per) * R + c]);
          if (k > k1 || fi > fimg || (fi == fimg && e < be)) {
            k1 = k;
            fimg = fi;
            be = e;
          }
        }
      }
      const uint32_t m1 = __reduce_max_sync(0xffffffffu, k1);
      const uint32_t mf = __reduce_max_sync(0xffffffffu, k1 == m1 ? fimg : 0u);
      const int me = int(__reduce_min_sync(0xffffffffu, k1 == m1 && fimg == mf ? uint32_t(be) : 0x7fffffffu));
      if (lane == 0) {
        s.choice[c] = m1 != 0u ? me : -1;
        s.key1[c] = m1;
        s.key2[c] = ((unsigned long long)mf << 6) | (unsigned long long)(63 - c);
      }
    }
    __syncthreads();
    // Arbitration: per expert the best (tokens, same node), then among those
    // the best (flow, lower rank).
    const int c = tid;
    const int ce = c < R ? s.choice[c] : -1;
    if (ce >= 0) atomicMax(&s.win1[ce], s.key1[c]);
    __syncthreads();
    if (ce >= 0 && s.win1[ce] == s.key1[c]) atomicMax(&s.win2[ce], s.key2[c]);
    __syncthreads();
    const bool winner = ce >= 0 && s.win1[ce] == s.key1[c] && s.win2[ce] == s.key2[c];
    const int h = ce >= 0 ? ce / per : 0;
    if (winner) atomicOr(&s.hmask[h], 1ull << c);
    if (ce >= 0) atomicAdd(s.any, 1);
    __syncthreads();
    // The winners' moves: ascending rank order on each home rank, home ranks in parallel.
    int pos = 0;
    if (winner) {
      const unsigned long long m = s.hmask[h];
      pos = __popcll(m & ((1ull << c) - 1ull));
      atomicMax(s.steps, __popcll(m));
    }
    __syncthreads();
    const int steps = *s.steps;
    for (int j = 0; j < steps; ++j) {
      if (winner && pos == j) {
        const int x = moved(s, R, per, words, total, fl, cl, c, ce);
        if (x > 0) {
          s.load[h] -= x;
          s.load[c] += x;
          s.w_rem[ce] -= x;
          s.used[c * words + (ce >> 5)] |= 1u << (ce & 31);
          se[c * K + s.n_slots[c]] = ce;
          st[c * K + s.n_slots[c]] = x;
          s.n_slots[c] += 1;
        }
      }
      __syncthreads();
    }
    // clear this round's arbitration state
    if (ce >= 0) {
      s.win1[ce] = 0u;
      s.win2[ce] = 0ull;
    }
    if (c < R) s.hmask[c] = 0ull;
    const bool any = *s.any != 0;
    __syncthreads();
    if (!any) break;
  }
  for (int r = tid; r < R; r += blockDim.x) p.rank_load[(long long)b * R + r] = int32_t(s.load[r]);
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
