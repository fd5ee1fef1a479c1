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
// The forward is one launch: every CTA streams rows of its grid-stride share,
// publishes its per-expert counts and sums of p, and the CTA that counts
// itself done last (no waiting: the others have already left) adds the
// partials up in a fixed order and writes the per-expert outputs, the batch
// scalars and the updated bias.  The backward is a plain streaming kernel.
#pragma once

#include "router_kernels.cuh"

namespace moe {

constexpr int kExtFwdThreads = 512;                   // one CTA per SM
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
  int32_t* tile_hist;          // workspace [E][G_stride]: per-CTA counts
  float* P_part;               // workspace [E][G_stride]: per-CTA sums of p
  int G_stride;
  unsigned long long* done;    // workspace counter of finished CTAs (zero between launches)
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
// col_of(v, l, i) (the layout of router_kernels.cuh).  Selection keys are
// 64-bit: the order-preserving image of the fp32 score z + b above the
// inverted column, so the group maximum is the largest score and, among equal
// scores, the lowest column.  k rounds each take the group maximum of the
// keys below the previous pick.
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV>
struct ExtRow {
  static constexpr int EPL = VW * NV;
  using Raw = typename DT::Raw;

  // Softmax statistics of the unbiased row: e[i] = 2^(z_i log2e - max log2e), inv_s = 1 / sum e.
  static __device__ __forceinline__ void softmax(const Raw (&raw)[EPL], bool valid, float (&e)[EPL], float& inv_s) {
    float m = -3.402823466e38f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, __uint_as_float(DT::bits(raw[i])));
    const float mL = group_max<LPR>(m) * kLog2e;
    row_exp<DT, LPR, EPL>(raw, mL, e);
    const float s = group_sum<LPR>(tree_sum(e));
    inv_s = valid ? rcp_approx(s) : 0.f;
  }

  // Top-k on z + b.  Returns the lane's own pick (lane j < k: pick j) with its
  // e, the sum of the picks' e, and the mask of the lane's picked elements.
  static __device__ __forceinline__ void select(const Raw (&raw)[EPL], const float (&bl)[EPL], const float (&e)[EPL],
                                                int k, int l, int& my_col, float& my_e, float& pick_sum,
                                                uint32_t& taken) {
    long long key[EPL];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        const float sv = __fadd_rn(__uint_as_float(DT::bits(raw[v * VW + i])), bl[v * VW + i]);
        key[v * VW + i] = Fp32::key_from_bits(__float_as_uint(sv), col_lane_bits<LPR, VW>(l), col_elem_bits<LPR, VW>(v, i));
      }
    long long prev = 0x7fffffffffffffffll;
    taken = 0u;
    pick_sum = 0.f;
    my_col = 0;
    my_e = 0.f;
    for (int j = 0; j < k; ++j) {
      long long lk = Fp32::kKeyMin;
#pragma unroll
      for (int i = 0; i < EPL; ++i) lk = (key[i] < prev && key[i] > lk) ? key[i] : lk;
      const long long w = group_max_key<LPR>(lk);
      float le = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const bool hit = key[i] == w;
        le = hit ? e[i] : le;
        taken |= hit ? (1u << i) : 0u;
      }
      const float pe = group_sum<LPR>(le);          // the winner's e; every other lane adds 0
      pick_sum += pe;
      if (l == j) {
        my_col = Fp32::key_col(w);
        my_e = pe;
      }
      prev = w;
    }
  }
};

// The per-expert outputs, the batch scalars and the updated bias, by the CTA
// that finished last.  Warp w adds up experts w, w + warps, ...: lane l the
// CTAs l, l + 32, ... (a fixed order), then a fixed shuffle tree, so the
// result does not depend on which CTA finishes last.  s_cnt / s_pe are the
// CTA's own shared arrays (its partials are already published).
__device__ __forceinline__ void ext_finalize(const FwdExParams& p, int G, int* s_cnt, float* s_pe) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = int(blockDim.x >> 5);
  for (int e = warp; e < p.E; e += nwarps) {
    const int32_t* hc = p.tile_hist + (long long)e * p.G_stride;
    const float* pc = p.P_part + (long long)e * p.G_stride;
    int c = 0;
    float s = 0.f;
    for (int b = lane; b < G; b += kWarp) {
      c += __ldcg(hc + b);
      s += __ldcg(pc + b);
    }
    c = __reduce_add_sync(0xffffffffu, c);
    s = warp_sum_f(s);
    if (lane == 0) {
      s_cnt[e] = c;
      s_pe[e] = s;
    }
  }
  __syncthreads();
  const long long TK = p.T * p.k;
  const double p_den = p.masked_p ? double(TK) : double(p.T);
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    const int c = s_cnt[e];
    p.counts[e] = c;
    p.f[e] = float(double(c) / double(TK));
    p.P[e] = float(double(s_pe[e]) / p_den);
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
      const float Pe = float(double(s_pe[e]) / p_den);
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
      *p.done = 0ull;                      // every CTA has counted itself: ready for the next launch
    }
  }
}

template <class DT, int LPR, int VW, int NV>
__global__ void __launch_bounds__(kExtFwdThreads, 1) router_fwd_ex_kernel(const FwdExParams p) {
  using Row = ExtRow<DT, LPR, VW, NV>;
  using Raw = typename DT::Raw;
  constexpr int EPL = Row::EPL;
  constexpr int GPW = kWarp / LPR;
  constexpr int COLS = LPR * VW * NV;
  static_assert(EPL <= 32, "taken mask");
  __shared__ float s_bias[COLS];
  __shared__ int s_hist[COLS];
  __shared__ float s_p[COLS];
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
    float e[EPL], inv_s;
    Row::softmax(raw, valid, e, inv_s);
    int my_col;
    float my_e, pick_sum;
    uint32_t taken;
    Row::select(raw, bl, e, p.k, l, my_col, my_e, pick_sum, taken);
    if (valid && l < p.k) {
      const long long a = t * p.k + l;
      p.idx[a] = my_col;
      p.gate[a] = p.renorm ? my_e * rcp_approx(pick_sum) : my_e * inv_s;
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
  const long long G = gridDim.x;
  for (int c = threadIdx.x; c < p.E; c += blockDim.x) {
    p.tile_hist[(long long)c * p.G_stride + blockIdx.x] = s_hist[c];
    p.P_part[(long long)c * p.G_stride + blockIdx.x] = s_p[c];
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(p.done, 1ull) == (unsigned long long)(G - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  ext_finalize(p, int(G), s_hist, s_p);
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
__global__ void __launch_bounds__(kExtBwdThreads) router_bwd_full_kernel(const BwdFullParams p) {
  using Raw = typename DT::Raw;
  constexpr int EPL = VW * NV;
  constexpr int RPW = kWarp / LPR;
  constexpr int COLS = LPR * VW * NV;
  __shared__ float s_f[COLS];
  for (int c = threadIdx.x; c < COLS; c += blockDim.x) s_f[c] = c < p.E ? __ldg(p.f + c) : 0.f;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int g = lane / LPR, l = lane % LPR;
  const long long gw = (long long)blockIdx.x * (kExtBwdThreads / kWarp) + (threadIdx.x >> 5);
  const long long nw = (long long)gridDim.x * (kExtBwdThreads / kWarp);
  const Raw* X = static_cast<const Raw*>(p.logits);
  const bool need_picks = p.dgate != nullptr || p.masked_p;
  float fr[EPL];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; ++i) fr[v * VW + i] = p.coef * s_f[col_of<LPR, VW>(v, l, i)];
  for (long long base = gw * RPW; base < p.T; base += nw * RPW) {
    const long long t = base + g;
    const bool valid = t < p.T;
    const Raw* row = X + (valid ? t : 0) * (long long)p.E;
    Raw raw[EPL];
    load_lane<DT, LPR, VW, NV, true>(row, p.E, l, valid, raw);
    // lane j < k of the group loads pick j and its upstream gradient
    const bool owner = need_picks && valid && l < p.k;
    int my_idx = -1;
    float my_dg = 0.f;
    if (owner) {
      my_idx = __ldg(p.idx + t * p.k + l);
      if (p.dgate != nullptr) my_dg = __ldg(p.dgate + t * p.k + l);
    }
    float m = -3.402823466e38f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, __uint_as_float(DT::bits(raw[i])));
    const float mL = group_max<LPR>(m) * kLog2e;
    float e[EPL];
    row_exp<DT, LPR, EPL>(raw, mL, e);
    const float s = group_sum<LPR>(tree_sum(e));
    const float inv_s = rcp_approx(s);
    // G of the lane's own pick
    float my_G = 0.f;
    if (p.dgate != nullptr) {
      if (p.renorm) {
        // e of the lane's pick, by the formula of row_exp (the same bits as its owner's e)
        Raw zr[1] = {DT::kNegInf};
        if (owner && unsigned(my_idx) < unsigned(p.E)) zr[0] = row[my_idx];   // out-of-range picks read nothing
        float my_e[1];
        row_exp<DT, LPR, 1>(zr, mL, my_e);
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
    // the lane's picked elements (mask) and their G
    float mk[EPL], gg[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      mk[i] = 0.f;
      gg[i] = 0.f;
    }
    if (need_picks) {
      for (int j = 0; j < p.k; ++j) {
        const int cj = __shfl_sync(0xffffffffu, my_idx, g * LPR + j);
        const float Gj = __shfl_sync(0xffffffffu, my_G, g * LPR + j);
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int i = 0; i < VW; ++i) {
            const bool hit = col_of<LPR, VW>(v, l, i) == cj;
            mk[v * VW + i] = hit ? 1.f : mk[v * VW + i];
            gg[v * VW + i] = hit ? Gj : gg[v * VW + i];
          }
      }
    }
    float dp[EPL], pd[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      dp[i] = (p.masked_p ? fr[i] * mk[i] : fr[i]) + gg[i];
      pd[i] = e[i] * dp[i];
    }
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
