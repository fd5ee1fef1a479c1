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
// The forward with bias routing and masked P is the persistent kernel's
// extended mode (router_kernels.cuh, kModeFwdExt).  This file holds the full
// backward, a plain streaming kernel, and the statistics of the shard combine
// (ext_outputs, which writes the per-expert outputs, the batch scalars and the
// updated bias from totals in shared memory).
#pragma once

#include "router_kernels.cuh"

namespace moe {

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
