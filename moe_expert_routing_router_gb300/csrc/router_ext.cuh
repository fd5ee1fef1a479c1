// Router kernels for the method's next steps:
//
//   * aux-loss-free bias routing: top-k on s = fp32(z) + b_e (the bias moves
//     selection only; softmax, gates and P use the unbiased z), and the bias
//     update b_e <- b_e + gamma * sign(T*k/E - count_e) after the batch;
//   * the masked P_i variant: P_i = (1/(T*k)) * sum_t p[t,i] * [i picked by t];
//   * the full router backward: the main loss's upstream gradient of the k
//     gates (plain p, or p renormalised over the picks) through the gate and
//     the softmax, added to the closed-form gradient of the aux loss.
//
// The forward is one launch: every CTA streams rows of its grid-stride share
// and adds its per-expert counts and sums of p into workspace accumulators
// with integer atomics; the CTA that counts itself done last (no waiting: the
// others have already left) writes the per-expert outputs, the batch scalars
// and the updated bias, and clears the accumulators.  A CTA's sum of p enters
// as two integers, its fixed-point value split at 2^-20 and 2^-64, so the
// total is exact to 2^-64 whatever the order of the atomics: the result does
// not depend on scheduling.  The backward is a plain streaming kernel.
#pragma once

#include "router_kernels.cuh"

namespace moe {

constexpr int kExtFwdThreads = 256;                   // two or more CTAs per SM
constexpr int kExtFwdWarps = kExtFwdThreads / kWarp;
constexpr int kExtBwdThreads = 256;

struct FwdExParams {
  const void* logits;          // [T, E] fp32 or bf16
  long long T;
  int E, k;
  int renorm;                  // gate renormalised over the picks
  int masked_p;                // P over the picked experts only, divided by T*k
  const float* bias;           // [E] selection bias, or null (all zero)
  float alpha;
  int n_ranks;
  float gamma;                 // bias step
  float* bias_out;             // [E] updated bias (may alias bias), or null
  int32_t* idx;                // [T, k]
  float* gate;                 // [T, k]
  int32_t* counts;             // [E]
  float* f;                    // [E]
  float* P;                    // [E]
  float* scalars;              // [kNumScalars]
  int32_t* rank_load;          // [n_ranks] or null
  // workspace accumulators, zero between launches (the last CTA clears them)
  int32_t* acc_count;          // [E] counts
  unsigned long long* acc_hi;  // [E] sums of p: integer parts of (CTA sum) * 2^20
  unsigned long long* acc_lo;  // [E] and the remaining fraction * 2^44
  unsigned long long* done;    // counter of finished CTAs
};

struct BwdFullParams {
  const void* logits;          // [T, E]
  long long T;
  int E, k;
  const float* f;              // [E]
  float coef;                  // dL/dp of the aux loss per unit f: g*alpha*E/T, or g*alpha*E/(T*k) when masked
  int masked_p;
  const int32_t* idx;          // [T, k] picks (null only without dgate and unmasked)
  const float* dgate;          // [T, k] upstream gradient of the gates, or null
  int renorm;
  float* dlogits;              // [T, E] fp32
};

// ---------------------------------------------------------------------------
// Forward, the row part.  Lane l of a row group holds the row's columns
// col_of(v, l, i) (the layout of router_kernels.cuh), in ascending column
// order along its elements.  Selection works on the order-preserving 32-bit
// image of the fp32 score z + b; each of the k rounds takes the group maximum
// of the images, then the lowest column holding it (ties go to the lower
// expert index), and clears that element's image to 0 (below every score's
// image, -inf included): afterwards exactly the picked elements read 0.
// ---------------------------------------------------------------------------
template <int LPR>
__device__ __forceinline__ uint32_t group_min_u32(uint32_t x) {
  if constexpr (LPR == 32) {
    return __reduce_min_sync(0xffffffffu, x);
  } else {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x = min(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
  }
}

// Maximum / minimum of N values as a tree of three-input operations (short
// dependency chains).
template <int N, bool MAX>
__device__ __forceinline__ uint32_t tree3_u32(const uint32_t (&x)[N]) {
  uint32_t t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = x[i];
#pragma unroll
  for (int n = N; n > 1; n = (n + 2) / 3) {
#pragma unroll
    for (int i = 0; i < n / 3; ++i)
      t[i] = MAX ? __vimax3_u32(t[3 * i], t[3 * i + 1], t[3 * i + 2]) : __vimin3_u32(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    if (n % 3 == 2) t[n / 3] = MAX ? max(t[n - 2], t[n - 1]) : min(t[n - 2], t[n - 1]);
    if (n % 3 == 1) t[n / 3] = t[n - 1];
  }
  return t[0];
}

// Larger value, larger image; -0 is folded into +0 first.
__device__ __forceinline__ uint32_t ordered_image(float x) {
  const uint32_t b = __float_as_uint(__fadd_rn(x, 0.f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <class DT, int LPR, int VW, int NV>
struct ExtRow {
  static constexpr int EPL = VW * NV;
  using Raw = typename DT::Raw;

  // Softmax statistics of the unbiased row: e[i] = 2^((z_i - mx) log2e), inv_s = 1 / sum e.
  static __device__ __forceinline__ void softmax(const Raw (&raw)[EPL], bool valid, float (&e)[EPL], float& mx,
                                                 float& inv_s) {
    float m = -3.402823466e38f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, __uint_as_float(DT::bits(raw[i])));
    mx = group_max<LPR>(m);
    row_exp<DT, LPR, EPL>(raw, mx, e);
    const float s = group_sum<LPR>(tree_sum(e));
    inv_s = valid ? rcp_approx(s) : 0.f;
  }

  // Top-k on z + b, exact by construction (k passes over the lane's
  // elements): lane j < k receives pick j's column; hv[i] == 0 marks the
  // lane's picked elements.
  static __device__ __forceinline__ void select_exact(const Raw (&raw)[EPL], const float (&bl)[EPL], int k, int l,
                                                      uint32_t (&hv)[EPL], int& my_col) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) hv[i] = ordered_image(__fadd_rn(__uint_as_float(DT::bits(raw[i])), bl[i]));
    const uint32_t lane_bits = col_lane_bits<LPR, VW>(l);
    my_col = 0;
    for (int j = 0; j < k; ++j) {
      const uint32_t wv = group_max_key<LPR>(tree3_u32<EPL, true>(hv));
      uint32_t cand[EPL];
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VW; ++i)
          cand[v * VW + i] = hv[v * VW + i] == wv ? (lane_bits | col_elem_bits<LPR, VW>(v, i)) : 0xffffffffu;
      const uint32_t wc = group_min_u32<LPR>(tree3_u32<EPL, false>(cand));
      // the column fields are disjoint: wc - lane_bits is the element's field iff this lane holds wc
      const uint32_t d = wc - lane_bits;
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VW; ++i) hv[v * VW + i] = d == col_elem_bits<LPR, VW>(v, i) ? 0u : hv[v * VW + i];
      if (l == j) my_col = int(wc);
    }
  }

  // Top-k on z + b with a per-lane cache (the fast path).  A key holds the
  // score image's upper 22 bits above the inverted 10-bit column, so keys are
  // distinct and one group maximum per round names the pick.  Each lane keeps
  // its two largest keys; the lane that wins takes its second key up, and a
  // lane whose cache runs empty refills it from its keys below the last one
  // taken.  One more round finds the best key left.  The key order is the
  // score order except between scores that share their upper 22 bits, so the
  // row is redone by select_exact when two consecutive keys of the k + 1 have
  // equal upper bits whose scores differ (for bf16 logits and a zero bias the
  // upper bits hold the whole score and nothing is redone).  Returns false
  // when the row must be redone; else lane j < k receives pick j's column
  // and bit i of `taken` marks the lane's picked elements.
  static __device__ __forceinline__ bool select_fast(const Raw (&raw)[EPL], const float (&bl)[EPL], int k, int l,
                                                     int& my_col, uint32_t& taken) {
    const uint32_t lane_bits = col_lane_bits<LPR, VW>(l);
    uint32_t key[EPL];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        const uint32_t img = ordered_image(__fadd_rn(__uint_as_float(DT::bits(raw[v * VW + i])), bl[v * VW + i]));
        key[v * VW + i] = (img & 0xfffffc00u) | (1023u - (lane_bits | col_elem_bits<LPR, VW>(v, i)));
      }
    uint32_t h1, h2;
    top2_keys(key, 0xffffffffu, h1, h2);
    my_col = 0;
    uint32_t prev = 0, cv = 0, kth = 0;
    bool ok = true, have_cv = false;
    for (int j = 0; j <= k; ++j) {
      const uint32_t w = group_max_key<LPR>(h1);
      if (j > 0 && (w >> 10) == (prev >> 10) && w != 0u) {       // equal upper bits: the fine order decides
        ok = ok && (!have_cv || cv == (w >> 10));
        have_cv = true;
        cv = w >> 10;
      }
      prev = w;
      if (j == k) break;
      kth = w;
      if (l == j) my_col = int(1023u - (w & 1023u));
      const bool won = h1 == w;
      const uint32_t last = w;
      h1 = won ? h2 : h1;
      const bool refill = won && h2 == 0u;
      h2 = won ? 0u : h2;
      if (__any_sync(0xffffffffu, refill) && refill) top2_keys(key, last, h1, h2);
    }
    // Scores sharing the collided upper bits must all be equal (then the
    // column order is the score order): their smallest and largest image agree.
    const bool collided = __any_sync(0xffffffffu, have_cv);
    ok = __all_sync(0xffffffffu, ok);
    if (collided && ok) {
      uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const uint32_t img = ordered_image(__fadd_rn(__uint_as_float(DT::bits(raw[i])), bl[i]));
        const bool in = have_cv && (img >> 10) == cv;
        lo = in ? min(lo, img) : lo;
        hi = in ? max(hi, img) : hi;
      }
      const uint32_t glo = group_min_u32<LPR>(lo), ghi = group_max_key<LPR>(hi);
      ok = __all_sync(0xffffffffu, !have_cv || glo == ghi);
    }
    taken = 0u;
#pragma unroll
    for (int i = 0; i < EPL; ++i) taken |= key[i] >= kth ? (1u << i) : 0u;
    return ok;
  }

  // The two largest of the lane's keys below `below` (0 where there are none),
  // as a pairwise tree: merging sorted pairs (h1, l1) and (h2, l2) gives
  // (max(h1, h2), max(min(h1, h2), l1, l2)).
  static __device__ __forceinline__ void top2_keys(const uint32_t (&key)[EPL], uint32_t below, uint32_t& m1, uint32_t& m2) {
    uint32_t k2[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) k2[i] = key[i] < below ? key[i] : 0u;
    if constexpr (EPL == 1) {
      m1 = k2[0];
      m2 = 0u;
    } else {
      constexpr int N0 = (EPL + 1) / 2;
      uint32_t hi[N0], lo[N0];
#pragma unroll
      for (int i = 0; i < EPL / 2; ++i) {
        hi[i] = max(k2[2 * i], k2[2 * i + 1]);
        lo[i] = min(k2[2 * i], k2[2 * i + 1]);
      }
      if constexpr (EPL & 1) {
        hi[N0 - 1] = k2[EPL - 1];
        lo[N0 - 1] = 0u;
      }
#pragma unroll
      for (int n = N0; n > 1; n = (n + 1) / 2) {
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
          const uint32_t a = hi[2 * i], b = hi[2 * i + 1];
          hi[i] = max(a, b);
          lo[i] = __vimax3_u32(min(a, b), lo[2 * i], lo[2 * i + 1]);
        }
        if (n & 1) {
          hi[n / 2] = hi[n - 1];
          lo[n / 2] = lo[n - 1];
        }
      }
      m1 = hi[0];
      m2 = lo[0];
    }
  }
};

// The per-expert outputs, the batch scalars and the updated bias, by the CTA
// that finished last: the accumulated totals go to shared memory (s_cnt, and
// the sums of p in double in s_pe) and the accumulators are cleared for the
// next launch.
__device__ __forceinline__ void ext_outputs(const FwdExParams& p, const int* s_cnt, const double* s_pe);

__device__ __forceinline__ void ext_finalize(const FwdExParams& p, int* s_cnt, double* s_pe) {
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    s_cnt[e] = __ldcg(p.acc_count + e);
    const unsigned long long hi = __ldcg(p.acc_hi + e), lo = __ldcg(p.acc_lo + e);
    s_pe[e] = (double(hi) + double(lo) * 0x1p-44) * 0x1p-20;
    p.acc_count[e] = 0;
    p.acc_hi[e] = 0ull;
    p.acc_lo[e] = 0ull;
  }
  __syncthreads();
  ext_outputs(p, s_cnt, s_pe);
  if (threadIdx.x == 0) *p.done = 0ull;   // every CTA has counted itself: ready for the next launch
}

// counts, f, P, the scalars, the rank loads and the updated bias from the
// totals in shared memory (s_cnt, and the sums of p in s_pe).
__device__ __forceinline__ void ext_outputs(const FwdExParams& p, const int* s_cnt, const double* s_pe) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long TK = p.T * p.k;
  const double p_den = p.masked_p ? double(TK) : double(p.T);
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    const int c = s_cnt[e];
    p.counts[e] = c;
    p.f[e] = float(double(c) / double(TK));
    p.P[e] = float(s_pe[e] / p_den);
    if (p.bias_out != nullptr) {
      // sign(T*k/E - count) from the exact integer comparison of count * E with T * k
      const long long d = TK - (long long)c * p.E;
      const float step = d > 0 ? p.gamma : (d < 0 ? -p.gamma : 0.f);
      p.bias_out[e] = __fadd_rn(p.bias != nullptr ? p.bias[e] : 0.f, step);
    }
  }
  if (warp == 0) {
    double fp = 0.0, d2 = 0.0;
    int cmax = -1, cmin = 0x7fffffff;
    for (int e = lane; e < p.E; e += kWarp) {
      const int c = s_cnt[e];
      const float fe = float(double(c) / double(TK));
      const float Pe = float(s_pe[e] / p_den);
      fp += double(fe) * double(Pe);
      const double d = double((long long)c * p.E - TK);
      d2 += d * d;
      cmax = max(cmax, c);
      cmin = min(cmin, c);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      fp += __shfl_xor_sync(0xffffffffu, fp, off);
      d2 += __shfl_xor_sync(0xffffffffu, d2, off);
    }
    cmax = __reduce_max_sync(0xffffffffu, cmax);
    cmin = __reduce_min_sync(0xffffffffu, cmin);
    // Per-rank loads: rank r hosts experts [r*E/R, (r+1)*E/R); lanes r and r + 32.
    const int R = p.n_ranks;
    double rd2 = 0.0;
    long long rmax = 0;
    for (int r = lane; r < R; r += kWarp) {
      const int per = p.E / R;
      long long load = 0;
      for (int e = r * per; e < (r + 1) * per; ++e) load += s_cnt[e];
      p.rank_load[r] = int32_t(load);
      const double d = double(load * R - TK);
      rd2 += d * d;
      rmax = load > rmax ? load : rmax;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      rd2 += __shfl_xor_sync(0xffffffffu, rd2, off);
      const long long o = __shfl_xor_sync(0xffffffffu, rmax, off);
      rmax = o > rmax ? o : rmax;
    }
    if (lane == 0) {
      const double balance = double(p.E) * fp;
      p.scalars[0] = float(double(p.alpha) * balance);
      p.scalars[1] = float(balance);
      p.scalars[2] = float(sqrt(d2 / double(p.E)) / double(TK));
      p.scalars[3] = float(double(cmax) * double(p.E) / double(TK));
      p.scalars[4] = float(double(cmin) * double(p.E) / double(TK));
      p.scalars[5] = R > 0 ? float(sqrt(rd2 / double(R)) / double(TK)) : 0.f;
      p.scalars[6] = R > 0 ? float(double(rmax) * double(R) / double(TK)) : 0.f;
    }
  }
}

// ---------------------------------------------------------------------------
// Combine the forward statistics of G shards of one batch (data-parallel ranks
// or slices routed one after another) into the batch's: counts summed exactly,
// P = sum_s P_s * T_s / T in double (the same for masked P, whose shard value
// divides by T_s * k), then f, the scalars and the rank loads as the forward
// computes them.  One CTA.
// ---------------------------------------------------------------------------
constexpr int kMaxShards = 64;

struct CombineParams {
  const int32_t* counts;       // [G, E]
  const float* P;              // [G, E]
  double T_shard[kMaxShards];  // tokens of each shard (passed by value)
  int G, E, k;
  long long T;                 // total tokens
  float alpha;
  int n_ranks;
  int masked_p;
  int32_t* counts_out;
  float* f;
  float* P_out;
  float* scalars;
  int32_t* rank_load;
};

cudaError_t launch_router_combine(const CombineParams& p, cudaStream_t stream);
cudaError_t launch_shard_capacity_base(const int32_t* counts, int G, int E, int rank, int32_t* base,
                                       cudaStream_t stream);

template <class DT, int LPR, int VW, int NV>
__global__ void __launch_bounds__(kExtFwdThreads, 2) router_fwd_ex_kernel(const FwdExParams p) {
  using Row = ExtRow<DT, LPR, VW, NV>;
  using Raw = typename DT::Raw;
  constexpr int EPL = Row::EPL;
  constexpr int GPW = kWarp / LPR;
  constexpr int COLS = LPR * VW * NV;
  __shared__ float s_bias[COLS];
  __shared__ int s_hist[COLS];
  __shared__ float s_p[COLS];
  __shared__ double s_pe[COLS];
  __shared__ int s_last;
  for (int c = threadIdx.x; c < COLS; c += blockDim.x) {
    s_bias[c] = (p.bias != nullptr && c < p.E) ? p.bias[c] : 0.f;
    s_hist[c] = 0;
    s_p[c] = 0.f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane / LPR, l = lane % LPR;
  float bl[EPL];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; ++i) bl[v * VW + i] = s_bias[col_of<LPR, VW>(v, l, i)];
  float pacc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) pacc[i] = 0.f;

  const Raw* X = static_cast<const Raw*>(p.logits);
  const long long n_rg = (p.T + GPW - 1) / GPW;              // row groups of GPW rows
  const long long nw = (long long)gridDim.x * kExtFwdWarps;
  long long rg = (long long)blockIdx.x * kExtFwdWarps + warp;
  // Software pipeline: the next row group's elements are loaded before the
  // current one is worked on.
  Raw nxt[EPL];
  {
    const long long t = rg * GPW + g;
    const bool ok = rg < n_rg && t < p.T;
    load_lane<DT, LPR, VW, NV, true>(X + (ok ? t : 0) * (long long)p.E, p.E, l, ok, nxt);
  }
  for (; rg < n_rg; rg += nw) {
    const long long t = rg * GPW + g;
    const bool valid = t < p.T;
    Raw raw[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) raw[i] = nxt[i];
    {
      const long long tn = (rg + nw) * GPW + g;
      const bool ok = rg + nw < n_rg && tn < p.T;
      load_lane<DT, LPR, VW, NV, true>(X + (ok ? tn : 0) * (long long)p.E, p.E, l, ok, nxt);
    }
    float e[EPL], mx, inv_s;
    Row::softmax(raw, valid, e, mx, inv_s);
    // The cached selection pays at 12 or more elements per lane (E = 384: 310 -> 276 us); with
    // fewer, its refills cost more than the passes they save (E = 64: 22 -> 24 us, E = 256: 137 -> 148 us).
    int my_col;
    uint32_t taken;
    if (EPL < 12 || !__all_sync(0xffffffffu, Row::select_fast(raw, bl, p.k, l, my_col, taken))) {
      uint32_t hv[EPL];
      Row::select_exact(raw, bl, p.k, l, hv, my_col);
      taken = 0u;
#pragma unroll
      for (int i = 0; i < EPL; ++i) taken |= hv[i] == 0u ? (1u << i) : 0u;
    }
    // The pick's e by the formula of row_exp from its logit (the same bits as
    // its owner's e[i]); the row was just read, so the load hits L1.
    const bool owner = valid && l < p.k;
    Raw zr[1] = {DT::kNegInf};
    if (owner) zr[0] = X[t * (long long)p.E + my_col];
    float my_e[1];
    row_exp<DT, LPR, 1>(zr, mx, my_e);
    const float pick_sum = owners_sum<LPR>(my_e[0]);
    if (owner) {
      const long long a = t * p.k + l;
      p.idx[a] = my_col;
      p.gate[a] = p.renorm ? my_e[0] * rcp_approx(pick_sum) : my_e[0] * inv_s;
      atomicAdd(&s_hist[my_col], 1);
    }
    if (p.masked_p) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) pacc[i] = ((taken >> i) & 1u) ? fmaf(e[i], inv_s, pacc[i]) : pacc[i];
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i) pacc[i] = fmaf(e[i], inv_s, pacc[i]);
    }
  }

  // The warp's sums of p per column (lanes with the same l), then the CTA's,
  // added warp by warp in a fixed order.
#pragma unroll
  for (int off = LPR; off < kWarp; off <<= 1)
#pragma unroll
    for (int i = 0; i < EPL; ++i) pacc[i] += __shfl_xor_sync(0xffffffffu, pacc[i], off);
  for (int w = 0; w < kExtFwdWarps; ++w) {
    if (warp == w && g == 0) {
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VW; ++i) {
          const int c = col_of<LPR, VW>(v, l, i);
          if (c < p.E) s_p[c] += pacc[v * VW + i];
        }
    }
    __syncthreads();
  }
  for (int c = threadIdx.x; c < p.E; c += blockDim.x) {
    if (s_hist[c] != 0) atomicAdd(p.acc_count + c, s_hist[c]);
    const double q = double(s_p[c]) * 0x1p20;          // s_p >= 0, below 2^31: q < 2^51
    const double hi = floor(q);
    const unsigned long long lo = (unsigned long long)((q - hi) * 0x1p44);   // exact for s_p >= 2^-41
    if (hi != 0.0) atomicAdd(p.acc_hi + c, (unsigned long long)hi);
    if (lo != 0ull) atomicAdd(p.acc_lo + c, lo);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(p.done, 1ull) == (unsigned long long)(gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  ext_finalize(p, s_hist, s_pe);
}

// ---------------------------------------------------------------------------
// Full backward of one row:
//   dp_i = A_i + G_i,   dz_i = p_i * (dp_i - sum_j p_j dp_j)
// with the aux part A_i = coef * f_i (unmasked P) or coef * f_i * m_i (masked
// P, coef then divides by T*k), and the gate part, for the picked experts
// (m_i = 1, dg_i the upstream gradient of the pick's gate):
//   G_i = dg_i                                (gate = p)
//   G_i = (dg_i - D) / S,  D = sum_j gate_j dg_j,  S = sum of the picks' p
//                                             (gate = p / S)
// Since the renormalised gates sum to 1, dg_i - D = sum_j gate_j (dg_i - dg_j);
// with e = p * s (s the row sum of e) and Se the picks' e:
//   G_i = s / Se^2 * sum_j e_j (dg_i - dg_j).
// That form takes each difference of two upstream gradients exactly once
// instead of subtracting their weighted mean, so close dg values lose no
// digits.  Lane j < k of the row group holds pick j (its column, dg and e);
// the k picks' e and dg go to every lane by shuffles.
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV>
__global__ void __launch_bounds__(kExtBwdThreads, (VW * NV <= 8 ? 5 : (VW * NV <= 12 ? 4 : 1))) router_bwd_full_kernel(const BwdFullParams p) {
  using Raw = typename DT::Raw;
  constexpr int EPL = VW * NV;
  constexpr int RPW = kWarp / LPR;
  constexpr int COLS = LPR * VW * NV;
  constexpr int WARPS = kExtBwdThreads / kWarp;
  __shared__ float s_f[COLS];
  // Per warp and row group: the picks' gradient terms scattered to their
  // columns (zero elsewhere; every pick's slot is cleared after use).
  __shared__ __align__(16) float s_g[WARPS][RPW][COLS];
  for (int c = threadIdx.x; c < COLS; c += blockDim.x) s_f[c] = c < p.E ? __ldg(p.f + c) : 0.f;
  for (int c = threadIdx.x; c < WARPS * RPW * COLS; c += blockDim.x) (&s_g[0][0][0])[c] = 0.f;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane / LPR, l = lane % LPR;
  const long long gw = (long long)blockIdx.x * WARPS + warp;
  const long long nw = (long long)gridDim.x * WARPS;
  const Raw* X = static_cast<const Raw*>(p.logits);
  const bool need_picks = p.dgate != nullptr || p.masked_p;
  float* sg = s_g[warp][g];
  float fr[EPL];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; ++i) fr[v * VW + i] = p.masked_p ? 0.f : p.coef * s_f[col_of<LPR, VW>(v, l, i)];
  // Software pipeline at 12 or more elements per lane: the next row group's
  // elements are loaded before the current one is worked on (the picks and
  // upstream gradients are not: their registers would cost a CTA per SM).
  // E = 384: 135 -> 128 us; at E = 64 it cost 1.3 us and is left out.
  constexpr bool kPrefetch = EPL >= 12;
  Raw nraw[EPL];
  if constexpr (kPrefetch) {
    const long long t0 = gw * RPW + g;
    const bool ok = gw * RPW < p.T && t0 < p.T;
    load_lane<DT, LPR, VW, NV, true>(X + (ok ? t0 : 0) * (long long)p.E, p.E, l, ok, nraw);
  }
  for (long long base = gw * RPW; base < p.T; base += nw * RPW) {
    const long long t = base + g;
    const bool valid = t < p.T;
    const Raw* row = X + (valid ? t : 0) * (long long)p.E;
    Raw raw[EPL];
    if constexpr (kPrefetch) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) raw[i] = nraw[i];
      const long long tn = base + nw * RPW + g;
      const bool ok = base + nw * RPW < p.T && tn < p.T;
      load_lane<DT, LPR, VW, NV, true>(X + (ok ? tn : 0) * (long long)p.E, p.E, l, ok, nraw);
    } else {
      load_lane<DT, LPR, VW, NV, true>(row, p.E, l, valid, raw);
    }
    // lane j < k of the group loads pick j and its upstream gradient
    const bool owner = need_picks && valid && l < p.k;
    int my_idx = 0;
    float my_dg = 0.f;
    if (owner) {
      my_idx = __ldg(p.idx + t * p.k + l);
      if (p.dgate != nullptr) my_dg = __ldg(p.dgate + t * p.k + l);
    }
    const bool in_range = owner && unsigned(my_idx) < unsigned(p.E);   // out-of-range picks touch nothing
    float m = -3.402823466e38f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, __uint_as_float(DT::bits(raw[i])));
    const float mx = group_max<LPR>(m);
    float e[EPL];
    row_exp<DT, LPR, EPL>(raw, mx, e);
    const float s = group_sum<LPR>(tree_sum(e));
    const float inv_s = rcp_approx(s);
    // The gradient term of the lane's own pick: the masked aux term and G.
    float my_G = 0.f;
    if (p.dgate != nullptr) {
      if (p.renorm) {
        // e of the lane's pick, by the formula of row_exp (the same bits as its owner's e)
        Raw zr[1] = {DT::kNegInf};
        if (in_range) zr[0] = row[my_idx];
        float my_e[1];
        row_exp<DT, LPR, 1>(zr, mx, my_e);
        float Se = 0.f, acc = 0.f;
        for (int j = 0; j < p.k; ++j) {
          const float ej = __shfl_sync(0xffffffffu, my_e[0], g * LPR + j);
          const float dj = __shfl_sync(0xffffffffu, my_dg, g * LPR + j);
          Se += ej;
          acc = fmaf(ej, my_dg - dj, acc);
        }
        const float inv_Se = rcp_approx(Se);
        my_G = owner ? acc * (s * inv_Se) * inv_Se : 0.f;
      } else {
        my_G = my_dg;
      }
    }
    __syncwarp();                                   // the previous row's slots are cleared
    if (in_range) sg[my_idx] = (p.masked_p ? p.coef * s_f[my_idx] : 0.f) + my_G;
    __syncwarp();
    float dp[EPL], pd[EPL];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int c0 = col_of<LPR, VW>(v, l, 0);
      float gv[VW];
      if constexpr (VW % 4 == 0) {
#pragma unroll
        for (int h = 0; h < VW / 4; ++h) {
          const float4 q = *reinterpret_cast<const float4*>(sg + c0 + 4 * h);
          gv[4 * h] = q.x; gv[4 * h + 1] = q.y; gv[4 * h + 2] = q.z; gv[4 * h + 3] = q.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < VW; ++i) gv[i] = sg[c0 + i];
      }
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        dp[v * VW + i] = fr[v * VW + i] + gv[i];
        pd[v * VW + i] = e[v * VW + i] * dp[v * VW + i];
      }
    }
    __syncwarp();
    if (in_range) sg[my_idx] = 0.f;
    const float w = inv_s * group_sum<LPR>(tree_sum(pd));      // sum_j p_j dp_j
    if (valid) {
      float* out = p.dlogits + t * (long long)p.E;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c0 = col_of<LPR, VW>(v, l, 0);
        if (c0 < p.E) {
          float d[VW];
#pragma unroll
          for (int i = 0; i < VW; ++i) d[i] = (e[v * VW + i] * inv_s) * (dp[v * VW + i] - w);
          store_vec_f32<VW>(out + c0, d);
        }
      }
    }
  }
}

}  // namespace moe
