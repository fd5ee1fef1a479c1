// Router kernels: softmax + top-k + Switch balance statistics (forward), the
// closed-form gradient of the aux loss (backward) and the capacity-limited
// stable dispatch, as one persistent cooperative kernel with grid barriers
// between the phases, plus a plain streaming kernel for the backward alone.
//
// Row layout.  A row of E logits is held by a group of LPR consecutive lanes
// (LPR in {8, 16, 32}; a warp holds 32/LPR rows).  Lane l of the group owns
// NV vectors of VW consecutive columns: column(v, l, i) = v*LPR*VW + l*VW + i,
// so one vector index across the group is one contiguous LPR*VW-column span
// (coalesced loads and stores).  LPR >= 8 >= k lets lane j of the group own
// the row's j-th pick.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"

namespace moe {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
constexpr int kMaxK = 8;

enum : int { kModeFwd = 1, kModeDispatch = 2, kModeBwd = 4, kModeStep = kModeFwd | kModeDispatch | kModeBwd };

struct RouterParams {
  const void* logits;          // [T, E] fp32 or bf16
  const int32_t* idx_in;       // [T, k] assignments to dispatch (dispatch-only mode)
  long long T;
  int E, k;
  float alpha;
  int renorm;
  int n_ranks;
  int C;                       // expert capacity
  float grad_scale;
  // outputs (null when the mode does not produce them)
  int32_t* idx;                // [T, k]
  float* gate;                 // [T, k]
  int32_t* counts;             // [E]
  float* f;                    // [E]
  float* P;                    // [E]
  float* scalars;              // [kNumScalars]
  int32_t* rank_load;          // [n_ranks]
  float* dlogits;              // [T, E]
  int32_t* perm;               // [T*k]
  int32_t* slot;               // [T*k]
  int32_t* offsets;            // [E+1]
  int32_t* kept;               // [E]
  int32_t* n_dropped;          // [1]
  // workspace
  Ctrl* ctrl;
  int32_t* tile_hist;          // [E][G_stride]: per-CTA counts, then their exclusive prefix over CTAs
  float* P_part;               // [E][G_stride]: per-CTA sums of p
  int32_t* counts_ws;          // [E] counts when `counts` is not an output
  int G;                       // CTAs in the grid
  int G_stride;
  unsigned long long timeout_ns;
};

constexpr int kNumScalars = 7;

struct BwdParams {
  const void* logits;
  long long T;
  int E;
  const float* f;
  float coef;                  // grad_scale * alpha * E / T
  float* dlogits;
};

// ---------------------------------------------------------------------------
// Shared-memory layout of the persistent kernel (ints/floats, 4 bytes each):
//   s_red  [64]        reduction scratch (also 32 doubles; first, so 8-byte aligned)
//   s_hist [E]         per-CTA expert counts (phase A)
//   s_off  [E + 1]     expert offsets (phase C)
//   s_w    [kWarps*E]  per-warp P partials (phase A), per-warp ranks (phase C)
// ---------------------------------------------------------------------------
__host__ __device__ inline size_t router_smem_bytes(int E) {
  return sizeof(int) * (size_t(E) + size_t(E + 1) + size_t(kWarps) * E + 64);
}

// ---------------------------------------------------------------------------
// Vector loads / stores of VW elements.
// ---------------------------------------------------------------------------
template <int BYTES> struct VecT;
template <> struct VecT<2> { using T = uint16_t; };
template <> struct VecT<4> { using T = uint32_t; };
template <> struct VecT<8> { using T = uint2; };
template <> struct VecT<16> { using T = uint4; };

template <class Raw, int VW>
__device__ __forceinline__ void load_vec(const Raw* src, Raw (&dst)[VW]) {
  constexpr int BYTES = int(sizeof(Raw)) * VW;
  if constexpr (BYTES <= 16) {
    using V = typename VecT<BYTES>::T;
    union { V v; Raw r[VW]; } u;
    u.v = __ldg(reinterpret_cast<const V*>(src));
#pragma unroll
    for (int i = 0; i < VW; ++i) dst[i] = u.r[i];
  } else {
    constexpr int H = 16 / int(sizeof(Raw));
    static_assert(VW % H == 0, "vector width");
#pragma unroll
    for (int h = 0; h < VW / H; ++h) {
      union { uint4 v; Raw r[H]; } u;
      u.v = __ldg(reinterpret_cast<const uint4*>(src + h * H));
#pragma unroll
      for (int i = 0; i < H; ++i) dst[h * H + i] = u.r[i];
    }
  }
}

template <int VW>
__device__ __forceinline__ void store_vec_f32(float* dst, const float* src) {
  if constexpr (VW == 1) {
    __stcs(dst, src[0]);
  } else if constexpr (VW == 2) {
    __stcs(reinterpret_cast<float2*>(dst), make_float2(src[0], src[1]));
  } else {
#pragma unroll
    for (int h = 0; h < VW / 4; ++h)
      __stcs(reinterpret_cast<float4*>(dst) + h, make_float4(src[4 * h], src[4 * h + 1], src[4 * h + 2], src[4 * h + 3]));
  }
}

// Loads lane l's EPL elements of row t (zeros for invalid rows / columns).
template <class DT, int LPR, int VW, int NV>
__device__ __forceinline__ void load_row(const typename DT::Raw* X, long long t, int E, int l, bool valid,
                                         typename DT::Raw (&raw)[VW * NV]) {
  using Raw = typename DT::Raw;
  constexpr int SPAN = LPR * VW;
  const Raw* row = X + t * (long long)E;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int c0 = v * SPAN + l * VW;
    Raw tmp[VW];
    if (valid && c0 < E) {   // E % VW == 0 for VW > 1: the whole vector is in the row
      if constexpr (VW == 1) tmp[0] = __ldg(row + c0);
      else load_vec<Raw, VW>(row + c0, tmp);
    } else {
#pragma unroll
      for (int i = 0; i < VW; ++i) tmp[i] = Raw(0);
    }
#pragma unroll
    for (int i = 0; i < VW; ++i) raw[v * VW + i] = tmp[i];
  }
}

template <int LPR, int VW>
__device__ __forceinline__ int col_of(int v, int l, int i) { return v * LPR * VW + l * VW + i; }

// ---------------------------------------------------------------------------
// Phase A: forward over rows [r0, r1).  Writes idx and gate, counts picks into
// s_hist (shared atomics) and leaves this warp's sums of p in s_w[warp][:].
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV>
__device__ __forceinline__ void fwd_rows(const RouterParams& p, long long r0, long long r1,
                                         int* s_hist, float* s_w) {
  using Raw = typename DT::Raw;
  using Key = typename DT::Key;
  constexpr int EPL = VW * NV;
  constexpr int RPW = kWarp / LPR;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane / LPR, l = lane % LPR;
  const int E = p.E, k = p.k;
  const Raw* X = static_cast<const Raw*>(p.logits);

  float pacc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) pacc[i] = 0.f;

  for (long long base = r0 + (long long)warp * RPW; base < r1; base += (long long)kWarps * RPW) {
    const long long t = base + g;
    const bool valid = t < r1;
    Raw raw[EPL];
    load_row<DT, LPR, VW, NV>(X, t, E, l, valid, raw);

    Key key[EPL];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        const int c = col_of<LPR, VW>(v, l, i);
        key[v * VW + i] = c < E ? DT::key(raw[v * VW + i], c) : DT::kKeyMin;
      }

    // Top-k: k rounds of "largest key below the previous winner".
    Key win[kMaxK];
    Key prev = DT::kKeyMin;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      win[j] = DT::kKeyMin;
      if (j < k) {
        Key local = DT::kKeyMin;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const bool below = (j == 0) || (key[i] < prev);
          local = (below && key[i] > local) ? key[i] : local;
        }
        win[j] = group_max_key<LPR>(local);
        prev = win[j];
      }
    }

    // Softmax against the row max (= the value of the first pick).
    const float mL = DT::key_value(win[0]) * kLog2e;
    float e[EPL];
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        const int c = col_of<LPR, VW>(v, l, i);
        const float x = DT::to_float(raw[v * VW + i]);
        e[v * VW + i] = c < E ? ex2_approx(fmaf(x, kLog2e, -mL)) : 0.f;
        s += e[v * VW + i];
      }
    s = group_sum<LPR>(s);
    const float inv_s = valid ? 1.f / s : 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) pacc[i] = fmaf(e[i], inv_s, pacc[i]);

    // Lane j of the group owns pick j.
    Key mine = DT::kKeyMin;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) mine = (j == l) ? win[j] : mine;
    const bool owner = l < k;
    const float ej = owner ? ex2_approx(fmaf(DT::key_value(mine), kLog2e, -mL)) : 0.f;
    const float denom = p.renorm ? group_sum<LPR>(ej) : s;
    if (valid && owner) {
      const int col = DT::key_col(mine);
      const long long a = t * k + l;
      p.idx[a] = col;
      p.gate[a] = ej / denom;
      atomicAdd(&s_hist[col], 1);
    }
  }

  // Sum the row groups of the warp, then group 0 stores the warp's partials.
#pragma unroll
  for (int i = 0; i < EPL; ++i)
#pragma unroll
    for (int off = LPR; off < kWarp; off <<= 1) pacc[i] += __shfl_xor_sync(0xffffffffu, pacc[i], off);
  if (g == 0) {
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        const int c = col_of<LPR, VW>(v, l, i);
        if (c < E) s_w[warp * E + c] = pacc[v * VW + i];
      }
  }
}

// ---------------------------------------------------------------------------
// Backward over rows [r0, r1) with row groups striding by `stride` rows:
//   dlogits[t,j] = coef * p[t,j] * (f[j] - sum_i p[t,i] f[i])
// `f` is read through L2 (it may have been written earlier in this launch).
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV>
__device__ __forceinline__ void bwd_rows(const void* logits, int E, const float* f, float coef, float* dlogits,
                                         long long first, long long r1, long long stride) {
  using Raw = typename DT::Raw;
  constexpr int EPL = VW * NV;
  const int lane = threadIdx.x & 31;
  const int g = lane / LPR, l = lane % LPR;
  const Raw* X = static_cast<const Raw*>(logits);

  float fr[EPL];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; ++i) {
      const int c = col_of<LPR, VW>(v, l, i);
      fr[v * VW + i] = c < E ? __ldcg(f + c) : 0.f;
    }

  for (long long base = first; base < r1; base += stride) {
    const long long t = base + g;
    const bool valid = t < r1;
    Raw raw[EPL];
    load_row<DT, LPR, VW, NV>(X, t, E, l, valid, raw);
    float x[EPL];
    float m = -3.402823466e38f;
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        const int c = col_of<LPR, VW>(v, l, i);
        x[v * VW + i] = DT::to_float(raw[v * VW + i]);
        if (c < E) m = fmaxf(m, x[v * VW + i]);
      }
    m = group_max<LPR>(m);
    const float mL = m * kLog2e;
    float e[EPL];
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        const int c = col_of<LPR, VW>(v, l, i);
        e[v * VW + i] = c < E ? ex2_approx(fmaf(x[v * VW + i], kLog2e, -mL)) : 0.f;
        s += e[v * VW + i];
      }
    s = group_sum<LPR>(s);
    const float inv_s = 1.f / s;
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      e[i] *= inv_s;                       // p
      dot = fmaf(e[i], fr[i], dot);
    }
    dot = group_sum<LPR>(dot);
    if (valid) {
      float* out = dlogits + t * (long long)E;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int c0 = col_of<LPR, VW>(v, l, 0);
        if (c0 < E) {
          float d[VW];
#pragma unroll
          for (int i = 0; i < VW; ++i) d[i] = coef * e[v * VW + i] * (fr[v * VW + i] - dot);
          store_vec_f32<VW>(out + c0, d);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Block-wide helpers (kThreads threads).
// ---------------------------------------------------------------------------

// Exclusive scan of n ints in place (n <= 4 * kThreads); returns the total.
__device__ __forceinline__ int block_exclusive_scan(int* data, int n, int* s_red, bool global_src) {
  constexpr int PER = 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int v[PER];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int j = tid * PER + i;
    v[i] = j < n ? (global_src ? __ldcg(data + j) : data[j]) : 0;
    sum += v[i];
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  __syncthreads();
  if (lane == 31) s_red[warp] = incl;
  __syncthreads();
  int warp_base = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int t = s_red[w];
    warp_base += w < warp ? t : 0;
    total += t;
  }
  int run = warp_base + incl - sum;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int j = tid * PER + i;
    if (j < n) data[j] = run;
    run += v[i];
  }
  __syncthreads();
  return total;
}

__device__ __forceinline__ double block_sum_d(double x, double* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  __syncthreads();
  if (lane == 0) s_red[warp] = x;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += s_red[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ int block_max_i(int x, int* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = __reduce_max_sync(0xffffffffu, x);
  __syncthreads();
  if (lane == 0) s_red[warp] = x;
  __syncthreads();
  int t = s_red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) t = max(t, s_red[w]);
  __syncthreads();
  return t;
}

__device__ __forceinline__ int block_min_i(int x, int* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = __reduce_min_sync(0xffffffffu, x);
  __syncthreads();
  if (lane == 0) s_red[warp] = x;
  __syncthreads();
  int t = s_red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) t = min(t, s_red[w]);
  __syncthreads();
  return t;
}

// ---------------------------------------------------------------------------
// Phase C dispatch: stable ranks of this CTA's assignments [a0, a1).
// tile_hist[e][cta] holds the exclusive prefix of expert e's count over the
// CTAs before this one; s_off the expert offsets.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dispatch_scatter(const RouterParams& p, const int32_t* idx_src, int cta,
                                                 long long a0, long long a1, const int* s_off, int* s_w) {
  const int E = p.E, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long n = a1 - a0;
  const long long w_lo = a0 + n * warp / kWarps, w_hi = a0 + n * (warp + 1) / kWarps;
  int* wh = s_w + warp * E;
  for (int e = lane; e < E; e += kWarp) wh[e] = 0;
  __syncwarp();
  for (long long a = w_lo + lane; a < w_hi; a += kWarp) {
    const int e = min(max(__ldcg(idx_src + a), 0), E - 1);
    atomicAdd(&wh[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) {
    int run = __ldcg(p.tile_hist + (size_t)e * p.G_stride + cta);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = s_w[w * E + e];
      s_w[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (long long base = w_lo; base < w_hi; base += kWarp) {
    const long long a = base + lane;
    const bool act = a < w_hi;
    const unsigned mask = __ballot_sync(0xffffffffu, act);
    int e = 0, r = 0, lower = 0;
    unsigned peers = 0;
    if (act) {
      e = min(max(__ldcg(idx_src + a), 0), E - 1);
      peers = __match_any_sync(mask, e);
      lower = __popc(peers & lt);
      r = wh[e] + lower;
    }
    __syncwarp();
    if (act && lower == 0) wh[e] += __popc(peers);
    __syncwarp();
    if (act) {
      p.perm[s_off[e] + r] = int(a);
      p.slot[a] = r < p.C ? r : -1;
    }
  }
}

// ---------------------------------------------------------------------------
// The persistent kernel.  MODE selects the phases:
//   A: per-CTA counts (and, with kModeFwd, idx/gate and sums of p)
//   B: per-expert totals, exclusive prefixes over CTAs, f and P
//   C: dispatch scatter (kModeDispatch), backward (kModeBwd), and the E-sized
//      outputs written by CTA 0 (scalars, rank loads, offsets, kept, drops).
// Launched cooperatively with p.G CTAs of kThreads threads.
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV, int MODE>
__global__ void __launch_bounds__(kThreads) router_persistent_kernel(const RouterParams p) {
  extern __shared__ int smem[];
  const int E = p.E, k = p.k, G = p.G, cta = blockIdx.x, tid = threadIdx.x;
  int* s_red = smem;
  int* s_hist = s_red + 64;
  int* s_off = s_hist + E;
  int* s_w = s_off + E + 1;
  float* s_wf = reinterpret_cast<float*>(s_w);
  double* s_red_d = reinterpret_cast<double*>(s_red);

  const long long r0 = p.T * cta / G, r1 = p.T * (cta + 1) / G;
  const long long a0 = r0 * k, a1 = r1 * k;
  int32_t* counts_dst = (MODE & kModeFwd) ? p.counts : p.counts_ws;

  // ---- phase A
  for (int e = tid; e < E; e += kThreads) s_hist[e] = 0;
  for (int i = tid; i < kWarps * E; i += kThreads) s_w[i] = 0;
  __syncthreads();
  if constexpr ((MODE & kModeFwd) != 0) {
    fwd_rows<DT, LPR, VW, NV>(p, r0, r1, s_hist, s_wf);
  } else {
    for (long long a = a0 + tid; a < a1; a += kThreads) {
      const int e = min(max(__ldg(p.idx_in + a), 0), E - 1);
      atomicAdd(&s_hist[e], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) {
    p.tile_hist[(size_t)e * p.G_stride + cta] = s_hist[e];
    if constexpr ((MODE & kModeFwd) != 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) t += s_wf[w * E + e];
      p.P_part[(size_t)e * p.G_stride + cta] = t;
    }
  }
  if (!grid_barrier(p.ctrl, G, p.timeout_ns, s_red + 63)) return;

  // ---- phase B: experts cta, cta + G, ...
  for (int e = cta; e < E; e += G) {
    const int total = block_exclusive_scan(p.tile_hist + (size_t)e * p.G_stride, G, s_red, true);
    if constexpr ((MODE & kModeFwd) != 0) {
      float t = 0.f;
      for (int j = tid; j < G; j += kThreads) t += __ldcg(p.P_part + (size_t)e * p.G_stride + j);
      const double Ps = block_sum_d(double(t), s_red_d);
      if (tid == 0) {
        p.counts[e] = total;
        p.f[e] = float(double(total) / double(p.T * k));
        p.P[e] = float(Ps / double(p.T));
      }
    } else {
      if (tid == 0) counts_dst[e] = total;
    }
    __syncthreads();
  }
  if (!grid_barrier(p.ctrl, G, p.timeout_ns, s_red + 63)) return;

  // ---- phase C
  if constexpr ((MODE & kModeDispatch) != 0) {
    for (int e = tid; e < E; e += kThreads) s_off[e] = __ldcg(counts_dst + e);
    __syncthreads();
    const int total = block_exclusive_scan(s_off, E, s_red, false);
    if (tid == 0) s_off[E] = total;
    __syncthreads();
    dispatch_scatter(p, (MODE & kModeFwd) ? p.idx : p.idx_in, cta, a0, a1, s_off, s_w);
  }
  if constexpr ((MODE & kModeBwd) != 0) {
    constexpr int RPW = kWarp / LPR;
    const float coef = p.grad_scale * p.alpha * float(E) / float(p.T);
    bwd_rows<DT, LPR, VW, NV>(p.logits, E, p.f, coef, p.dlogits, r0 + (long long)(tid >> 5) * RPW, r1,
                              (long long)kWarps * RPW);
  }
  if (cta == 0) {
    if constexpr ((MODE & kModeDispatch) != 0) {
      __syncthreads();
      int dropped = 0;
      for (int e = tid; e <= E; e += kThreads) {
        p.offsets[e] = s_off[e];
        if (e < E) {
          const int c = __ldcg(counts_dst + e);
          p.kept[e] = min(c, p.C);
          dropped += max(c - p.C, 0);
        }
      }
      const double d = block_sum_d(double(dropped), s_red_d);
      if (tid == 0) *p.n_dropped = int(d);
    }
    if constexpr ((MODE & kModeFwd) != 0) {
      const double mean = double(p.T) * k / E;
      double fp = 0.0, dev = 0.0;
      int cmax = 0, cmin = 0x7fffffff;
      for (int e = tid; e < E; e += kThreads) {
        const int c = __ldcg(p.counts + e);
        fp += double(__ldcg(p.f + e)) * double(__ldcg(p.P + e));
        dev += (double(c) - mean) * (double(c) - mean);
        cmax = max(cmax, c);
        cmin = min(cmin, c);
      }
      fp = block_sum_d(fp, s_red_d);
      dev = block_sum_d(dev, s_red_d);
      cmax = block_max_i(cmax, s_red);
      cmin = block_min_i(cmin, s_red);
      double rdev = 0.0;
      int rmax = 0;
      const int R = p.n_ranks;
      if (R > 0) {
        const int per = E / R;
        const double rmean = double(p.T) * k / R;
        for (int r = tid; r < R; r += kThreads) {
          int load = 0;
          for (int j = 0; j < per; ++j) load += __ldcg(p.counts + r * per + j);
          p.rank_load[r] = load;
          rdev += (double(load) - rmean) * (double(load) - rmean);
          rmax = max(rmax, load);
        }
        rdev = block_sum_d(rdev, s_red_d);
        rmax = block_max_i(rmax, s_red);
      }
      if (tid == 0) {
        const double balance = double(E) * fp;
        p.scalars[0] = float(double(p.alpha) * balance);
        p.scalars[1] = float(balance);
        p.scalars[2] = float(sqrt(dev / E) / mean);
        p.scalars[3] = float(cmax / mean);
        p.scalars[4] = float(cmin / mean);
        if (R > 0) {
          const double rmean = double(p.T) * k / R;
          p.scalars[5] = float(sqrt(rdev / R) / rmean);
          p.scalars[6] = float(rmax / rmean);
        } else {
          p.scalars[5] = 0.f;
          p.scalars[6] = 0.f;
        }
      }
    }
  }
}

// Backward alone: a plain grid-stride streaming kernel.
template <class DT, int LPR, int VW, int NV>
__global__ void __launch_bounds__(kThreads) router_bwd_kernel(const BwdParams p) {
  constexpr int RPW = kWarp / LPR;
  const long long gw = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const long long nw = (long long)gridDim.x * kWarps;
  bwd_rows<DT, LPR, VW, NV>(p.logits, p.E, p.f, p.coef, p.dlogits, gw * RPW, p.T, nw * RPW);
}

}  // namespace moe
