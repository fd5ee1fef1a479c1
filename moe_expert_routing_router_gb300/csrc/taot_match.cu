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
// One CTA per microbatch.  Same node and flow depend only on the pair of ranks
// (h, c), so the best expert of c splits into a best per home rank h, by tokens
// and then the lower index, and a best over h by (tokens, same node, flow, lower
// index).  The CTA keeps the table best[h][c] in shared memory.  An entry
// changes only when a move touches h (its load and its experts' tokens left) or
// c (its load, its slots, the experts it already hosts), so after the first
// round only the rows and columns of the ranks that moved tokens are
// recomputed.  Each round then has three parts, separated by block barriers:
// the table update; the per-rank choice, eight warps each taking a quarter of
// the home ranks for 32 cold ranks; and, in warp 0 alone with warp-level
// synchronisation, the merge of the quarters, the arbitration and the commits.
// The arbitration is two shared-memory atomic maxima per expert over its
// choosers' keys, (tokens, same node) and then (flow, inverted rank), so the
// best chooser and, among equal ones, the lowest rank wins.  The winners' moves
// are committed in ascending rank order within each hot home rank (the only
// quantity two winners of a round share is the load of the hot rank they both
// draw on) and in parallel across home ranks.  floor((load * R - total) / R)
// is load - ceil(total / R) and floor((total - load * R) / R) is
// floor(total / R) - load, so no division is left in the scoring.
#include "taot_match.h"

namespace moe {
namespace {

constexpr int kMatchThreads = 256;   // eight warps: two blocks of 32 cold ranks x four quarters of the home ranks
constexpr int kParts = 4;

struct MatchSmem {
  long long* load;     // [R]
  long long* total;    // [1]
  unsigned long long* win2;   // [E] best key2 among the choosers with the best key1
  unsigned long long* hmask;  // [R] this round's winners drawing on hot home rank h, one bit per rank
  int32_t* w_rem;      // [E]
  uint32_t* used;      // [R][E / 32 rounded up]
  int32_t* n_slots;    // [R]
  uint32_t* win1;      // [E] best key1 among the expert's choosers this round (0: none)
  uint32_t* fimg;      // [R][R] order-preserving image of this microbatch's Phase 1 flow, [h][c]
  uint32_t* bk;        // [R][64] best (tokens << 1 | same node) of cold rank c on home rank h (0: none), at tab(h, c)
  uint16_t* be;        // [R][64] the expert of that entry
  uint32_t* pk;        // [kParts][R] per quarter of the home ranks: best key of cold rank c
  uint32_t* pf;        // [kParts][R] its flow image
  int32_t* pe;         // [kParts][R] its expert
  uint8_t* hl;         // [R] home ranks whose table rows are recomputed this round
  uint8_t* cl;         // [R] cold ranks whose table columns are recomputed this round
  int32_t* nh;         // [1] entries of hl
  int32_t* nc;         // [1] entries of cl
  int32_t* any;        // [1] the round had a choice (another round follows)
  unsigned long long* dh;     // [1] bit h: home rank h is in hl
};

__host__ __device__ inline size_t a16(size_t x) { return (x + 15) / 16 * 16; }

__host__ __device__ inline size_t match_layout(int E, int R, MatchSmem* s, char* base) {
  const int words = (E + 31) / 32;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off += a16(bytes); return base ? base + o : nullptr; };
  char* load = take(8u * R);
  char* total = take(8u);
  char* win2 = take(8u * E);
  char* hmask = take(8u * R);
  char* w_rem = take(4u * E);
  char* used = take(4u * R * words);
  char* n_slots = take(4u * R);
  char* win1 = take(4u * E);
  char* fimg = take(4u * R * R);
  char* bk = take(4u * R * 64);
  char* be = take(2u * R * 64);
  char* pk = take(4u * kParts * R);
  char* pf = take(4u * kParts * R);
  char* pe = take(4u * kParts * R);
  char* hl = take(1u * R);
  char* cl = take(1u * R);
  char* nh = take(4u);
  char* nc = take(4u);
  char* any = take(4u);
  char* dh = take(8u);
  if (s) {
    s->load = reinterpret_cast<long long*>(load);
    s->total = reinterpret_cast<long long*>(total);
    s->win2 = reinterpret_cast<unsigned long long*>(win2);
    s->hmask = reinterpret_cast<unsigned long long*>(hmask);
    s->w_rem = reinterpret_cast<int32_t*>(w_rem);
    s->used = reinterpret_cast<uint32_t*>(used);
    s->n_slots = reinterpret_cast<int32_t*>(n_slots);
    s->win1 = reinterpret_cast<uint32_t*>(win1);
    s->fimg = reinterpret_cast<uint32_t*>(fimg);
    s->bk = reinterpret_cast<uint32_t*>(bk);
    s->be = reinterpret_cast<uint16_t*>(be);
    s->pk = reinterpret_cast<uint32_t*>(pk);
    s->pf = reinterpret_cast<uint32_t*>(pf);
    s->pe = reinterpret_cast<int32_t*>(pe);
    s->hl = reinterpret_cast<uint8_t*>(hl);
    s->cl = reinterpret_cast<uint8_t*>(cl);
    s->nh = reinterpret_cast<int32_t*>(nh);
    s->nc = reinterpret_cast<int32_t*>(nc);
    s->any = reinterpret_cast<int32_t*>(any);
    s->dh = reinterpret_cast<unsigned long long*>(dh);
  }
  return off;
}

// Position of the table entry (h, c): rows of 64, columns swizzled by the row so
// that a warp reads or writes conflict-free both along a row (fixed h) and along
// a column (fixed c).
__device__ __forceinline__ int tab(int h, int c) { return h * 64 + (c ^ (h & 31)); }

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

// Best expert of home rank h for cold rank c as the state stands: the most
// tokens moved, then the lower index; the key is (tokens << 1) | same node.
__device__ __forceinline__ void update_entry(const MatchSmem& s, int R, int per, int words, int K, int rpn,
                                             long long total, long long fl, long long cl, int h, int c) {
  uint32_t bkey = 0u;
  int bexp = 0;
  const long long Lh = s.load[h], Lc = s.load[c];
  if (Lh * R > total && Lc * R < total && s.n_slots[c] < K) {
    const long long lim = Lh - cl < fl - Lc ? Lh - cl : fl - Lc;
    if (lim > 0) {
      const uint32_t same = h / rpn == c / rpn ? 1u : 0u;
      const uint32_t* urow = s.used + c * words;
      for (int e = h * per; e < (h + 1) * per; ++e) {
        const int wr = s.w_rem[e];
        if (wr <= 0 || ((urow[e >> 5] >> (e & 31)) & 1u)) continue;
        const long long x = wr < lim ? wr : lim;
        const uint32_t key = (uint32_t(x) << 1) | same;
        if (key > bkey) {
          bkey = key;
          bexp = e;
        }
      }
    }
  }
  s.bk[tab(h, c)] = bkey;
  s.be[tab(h, c)] = uint16_t(bexp);
}

// Keeps (k, f, e) if it beats the best so far: larger key, then larger flow
// image, then lower expert.
__device__ __forceinline__ void better(uint32_t k, uint32_t f, int e, uint32_t& k1, uint32_t& f1, int& e1) {
  if (k == 0u || k < k1) return;
  if (k > k1 || f > f1 || (f == f1 && e < e1)) {
    k1 = k;
    f1 = f;
    e1 = e;
  }
}

__global__ void __launch_bounds__(kMatchThreads) taot_match_kernel(const MatchParams p) {
  extern __shared__ __align__(16) char smem[];
  MatchSmem s;
  match_layout(p.E, p.R, &s, smem);
  const int b = blockIdx.x, R = p.R, E = p.E, K = p.K, per = E / R, words = (E + 31) / 32, rpn = p.ranks_per_node;
  const int32_t* w = p.expert_loads + (long long)b * E;
  const float* plan = p.plan + (long long)b * R * R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = kMatchThreads / 32;
  for (int e = tid; e < E; e += blockDim.x) {
    s.w_rem[e] = w[e];
    s.win1[e] = 0u;
    s.win2[e] = 0ull;
  }
  for (int i = tid; i < R * R; i += blockDim.x) s.fimg[i] = flow_image(plan[i]);
  for (int i = tid; i < R * words; i += blockDim.x) s.used[i] = 0u;
  for (int r = tid; r < R; r += blockDim.x) {
    s.n_slots[r] = 0;
    s.hmask[r] = 0ull;
    s.hl[r] = uint8_t(r);                          // the first round computes every row
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
    *s.nh = R;
    *s.nc = 0;
    *s.dh = R == 64 ? ~0ull : (1ull << R) - 1ull;
  }
  __syncthreads();
  const long long total = *s.total;
  const long long fl = total >= 0 ? total / R : -((-total + R - 1) / R);
  const long long cl = total >= 0 ? (total + R - 1) / R : -((-total) / R);
  const int hq = (R + kParts - 1) / kParts;
  // Rounds repeat while some cold rank still finds a positive match.  A round
  // with a choice commits at least its lowest-ranked winner (no earlier move of
  // the round changed its numbers), and a rank holds at most K replicas, so
  // there are at most R * K + 1 rounds.
  for (int round = 0; round <= R * K; ++round) {
    // Table update: the rows of the home ranks that gave tokens last round (all
    // of them before the first), then the columns of the cold ranks that took
    // tokens, without the entries the rows already covered.
    {
      const int nh = *s.nh, nc = *s.nc;
      const unsigned long long dh = *s.dh;
      for (int i = tid; i < (nh + nc) * 64; i += kMatchThreads) {
        int h, c;
        if (i < nh * 64) {
          h = s.hl[i >> 6];
          c = i & 63;
        } else {
          const int j = i - nh * 64;
          c = s.cl[j >> 6];
          h = j & 63;
          if (h < R && ((dh >> h) & 1ull)) continue;
        }
        if (h < R && c < R) update_entry(s, R, per, words, K, rpn, total, fl, cl, h, c);
      }
    }
    __syncthreads();
    // Per-rank choice over a quarter of the home ranks: warp w takes cold ranks
    // 32 (w & 1) + lane and the hot ones among home ranks
    // [hq (w >> 1), hq (w >> 1 + 1)) (a home rank that is not hot has no entry).
    {
      const int c = (warp & 1) * 32 + lane, part = warp >> 1;
      const unsigned hot_lo = __ballot_sync(0xffffffffu, lane < R && s.load[lane] * R > total);
      const unsigned hot_hi = __ballot_sync(0xffffffffu, lane + 32 < R && s.load[lane + 32] * R > total);
      const int h0 = part * hq, h1 = (part + 1) * hq < R ? (part + 1) * hq : R;
      unsigned long long m = ((unsigned long long)hot_hi << 32) | hot_lo;
      m &= (h1 == 64 ? ~0ull : (1ull << h1) - 1ull) & ~((1ull << h0) - 1ull);
      uint32_t k1 = 0u, f1 = 0u;
      int e1 = 0x7fffffff;
      for (; m != 0ull; m &= m - 1ull) {
        const int h = __ffsll((long long)m) - 1;
        const uint32_t k = c < R ? s.bk[tab(h, c)] : 0u;
        if (k != 0u && k >= k1) better(k, s.fimg[h * R + c], s.be[tab(h, c)], k1, f1, e1);
      }
      if (c < R) {
        s.pk[part * R + c] = k1;
        s.pf[part * R + c] = f1;
        s.pe[part * R + c] = e1;
      }
    }
    __syncthreads();
    // Warp 0 alone (lane l holds ranks l and l + 32): the merge of the quarters
    // into each rank's choice; the arbitration, per expert the best (tokens,
    // same node), then among those the best (flow, lower rank), by shared-memory
    // atomic maxima; the winners' moves, in ascending rank order on each hot
    // home rank and in parallel across home ranks; the lists of ranks whose
    // table entries change; the clearing of the round's arbitration state.
    if (warp == 0) {
      int ce[2], hh[2], pos[2];
      uint32_t ck1[2];
      unsigned long long ck2[2];
      bool win[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = lane + 32 * j;
        uint32_t k1 = 0u, f1 = 0u;
        int e1 = 0x7fffffff;
        if (c < R) {
#pragma unroll
          for (int q = 0; q < kParts; ++q) better(s.pk[q * R + c], s.pf[q * R + c], s.pe[q * R + c], k1, f1, e1);
        }
        ce[j] = k1 != 0u ? e1 : -1;
        ck1[j] = k1;
        ck2[j] = ((unsigned long long)f1 << 6) | (unsigned long long)(63 - c);
        if (ce[j] >= 0) atomicMax(&s.win1[ce[j]], k1);
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (ce[j] >= 0 && s.win1[ce[j]] == ck1[j]) atomicMax(&s.win2[ce[j]], ck2[j]);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = lane + 32 * j;
        win[j] = ce[j] >= 0 && s.win1[ce[j]] == ck1[j] && s.win2[ce[j]] == ck2[j];
        hh[j] = ce[j] >= 0 ? ce[j] / per : 0;
        if (win[j]) atomicOr(&s.hmask[hh[j]], 1ull << c);
      }
      __syncwarp();
      int steps = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = lane + 32 * j;
        pos[j] = 0;
        if (win[j]) {
          const unsigned long long m = s.hmask[hh[j]];
          pos[j] = __popcll(m & ((1ull << c) - 1ull));
          steps = max(steps, __popcll(m));
        }
      }
      steps = int(__reduce_max_sync(0xffffffffu, uint32_t(steps)));
      unsigned long long gave = 0ull, took = 0ull;   // this lane's commits: home ranks and cold ranks
      for (int step = 0; step < steps; ++step) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = lane + 32 * j;
          if (win[j] && pos[j] == step) {
            const int x = moved(s, R, per, words, total, fl, cl, c, ce[j]);
            if (x > 0) {
              s.load[hh[j]] -= x;
              s.load[c] += x;
              s.w_rem[ce[j]] -= x;
              s.used[c * words + (ce[j] >> 5)] |= 1u << (ce[j] & 31);
              se[c * K + s.n_slots[c]] = ce[j];
              st[c * K + s.n_slots[c]] = x;
              s.n_slots[c] += 1;
              gave |= 1ull << hh[j];
              took |= 1ull << c;
            }
          }
        }
        __syncwarp();
      }
      const bool any = __any_sync(0xffffffffu, ce[0] >= 0 || ce[1] >= 0);
      gave = (unsigned long long)__reduce_or_sync(0xffffffffu, uint32_t(gave)) |
             ((unsigned long long)__reduce_or_sync(0xffffffffu, uint32_t(gave >> 32)) << 32);
      took = (unsigned long long)__reduce_or_sync(0xffffffffu, uint32_t(took)) |
             ((unsigned long long)__reduce_or_sync(0xffffffffu, uint32_t(took >> 32)) << 32);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (ce[j] >= 0) {
          s.win1[ce[j]] = 0u;
          s.win2[ce[j]] = 0ull;
        }
        const int r = lane + 32 * j;
        if (r < R) s.hmask[r] = 0ull;
        const unsigned long long below = (1ull << r) - 1ull;
        if ((gave >> r) & 1ull) s.hl[__popcll(gave & below)] = uint8_t(r);
        if ((took >> r) & 1ull) s.cl[__popcll(took & below)] = uint8_t(r);
      }
      if (lane == 0) {
        *s.any = any ? 1 : 0;
        *s.nh = __popcll(gave);
        *s.nc = __popcll(took);
        *s.dh = gave;
      }
    }
    __syncthreads();
    if (*s.any == 0) break;                        // written before the barrier, rewritten only after the next two
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
