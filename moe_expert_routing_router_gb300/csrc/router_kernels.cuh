// Router kernels: softmax + top-k + Switch balance statistics (forward), the
// closed-form gradient of the aux loss (backward) and the capacity-limited
// stable dispatch, as one persistent cooperative kernel with one grid barrier
// between the forward and the rest, plus a plain streaming kernel for the
// backward alone.
//
// CTA organisation (one CTA per SM, kThreads = 640):
//   warps 0..17 consumers: the per-row forward and backward math (for a
//               dispatch of given assignments: the ranking and the scatter)
//   warp  18    producer: streams this CTA's contiguous chunk of logit rows
//               into a shared-memory ring with bulk asynchronous copies (TMA),
//               and refills it for the backward
//   warp  19    dispatcher: stable ranks of the forward's picks as they are
//               made, the sums of p of the CTA's experts, the scatter during
//               the backward, and (in the CTA that finishes its per-expert
//               outputs last) the E-sized outputs
//
// Row layout.  A row of E logits is held by a group of LPR consecutive lanes
// (LPR in {8, 16, 32}; a warp holds 32/LPR rows).  Lane l of the group owns
// NV vectors of VW consecutive columns: column(v, l, i) = v*LPR*VW + l*VW + i,
// so one vector index across the group is one contiguous LPR*VW-column span.
// LPR >= 8 >= k lets lane j of the group own the row's j-th pick.
//
// Ring.  Stage s of the chunk (rows_per_stage rows) goes to slot s % n_slots.
// The backward walks the stages in reverse: the last n_slots stages of the
// forward are still in the ring and are used without reloading; older stages
// are reloaded into the slot freed by the stage n_slots above them.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"

namespace moe {

// One CTA per SM: 18 consumer warps, one producer (TMA) warp, one dispatch
// warp -- five warps on each of the SM's four schedulers.  The consumers share
// one ring, so a warp the scheduler favours cannot run more than the ring's
// depth ahead of the others.  (Five warps per scheduler cap a thread at 96
// registers.)
constexpr int kConsumerWarps = 18;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kDispatchWarp = kConsumerWarps + 1;
constexpr int kThreads = (kConsumerWarps + 2) * kWarp;
constexpr int kConsumerThreads = kConsumerWarps * kWarp;
// Consumers + producer: the CTA-level syncs from the end of the forward to the
// start of the backward exclude the dispatch warp, whose in-CTA ranking runs
// on through the grid barrier and the totals.
constexpr int kMainThreads = (kConsumerWarps + 1) * kWarp;
static_assert(kMainThreads / kWarp <= 32, "block scans hold one value per warp in 32 slots");
// Slots of the 128-int scratch area at the start of shared memory.
constexpr int kRedProg = 64;     // forward stages finished, per consumer warp
constexpr int kRedPhase = 96;    // 1 once the grid barrier has passed, 2 once this CTA's totals, bases and
                                 // offsets are in shared memory, -1 after an error
constexpr int kRedRanked = 97;   // 1 once the dispatch warp has ranked every pick of the CTA, -1 if it gave up
constexpr int kRedFixNext = 98;  // next chunk of the CTA's final dispatch positions to write
constexpr int kRedFlag = 127;    // grid barrier result
// The candidate set of the fast top-k path (see fwd_groups_fast): 64 columns
// in the 128-int scratch (two per lane, 16 bits each in 32 ints), their
// membership bitmap (E <= 1024 bits) and a flag set once both are written.
constexpr int kRedCand = 0;
constexpr int kRedCandBits = 32;
constexpr int kRedCandReady = 99;
constexpr int kRedBwdLast = 100;  // a split step: 1 in the CTA that added its sums of p last
constexpr int kRedCandDone = 101; // consumer warps that have added their columns of the first stage
static_assert(kConsumerWarps <= 32, "progress slots");
constexpr int kBarMain = 2;       // named barrier of the main group
constexpr int kBarConsumers = 1;  // named barrier of the consumer warps
constexpr int kMaxK = 8;
// The final dispatch positions of a CTA's picks are written in chunks of this
// many assignments: by the dispatch warp while the consumers run the backward,
// and by the consumers that have finished it.
constexpr int kFixupChunk = 256;
constexpr int kCtrlNoExpert = 1 << 16;   // above every expert id (dispatch peer matching)
constexpr int kGridMax = 1024;   // CTAs of a persistent launch at most (the per-CTA partial tables' width)
constexpr int kGroupCtas = 8;    // CTAs per group of the per-group count sums
constexpr int kGroupMax = kGridMax / kGroupCtas;
constexpr int kMaxSlots = 16;
constexpr int kMaxExperts = 1024;
constexpr int kNumScalars = 7;
// Limit of the wait for this CTA's own bulk copies before it exits; it does not
// follow RouterParams::timeout_ns, which tests shorten.
constexpr unsigned long long kDrainNs = 1000000000ull;

// kModeSplit (with kModeStep, renormalised gates): the forward takes only the
// top-k and the gates; the backward forms each row's softmax sum and P.
// kModeExt: the extended step (with kModeStep) -- selection on fp32(z) + b,
// masked P when asked, the bias update, and the backward of the gates' upstream
// gradient added to the aux loss's -- or its forward alone (with kModeFwd).
enum : int {
  kModeFwd = 1, kModeDispatch = 2, kModeBwd = 4, kModeSplit = 8, kModeExt = 16,
  kModeStep = kModeFwd | kModeDispatch | kModeBwd, kModeStepSplit = kModeStep | kModeSplit,
  kModeStepExt = kModeStep | kModeExt, kModeFwdExt = kModeFwd | kModeExt
};

// The type of the pick slots: the 32-bit selection keys of the biased scores
// in the extended step, the element type's keys otherwise.
template <bool EXT, class Key> struct PickKeyOf { using type = Key; };
template <class Key> struct PickKeyOf<true, Key> { using type = uint32_t; };

struct RouterParams {
  const void* logits;          // [T, E] fp32 or bf16
  const int32_t* idx_in;       // [T, k] assignments to dispatch (dispatch-only mode)
  long long T;
  int E, k;
  float alpha;
  int renorm;
  int n_ranks;
  int C;                       // expert capacity
  const int32_t* cap_base;     // [E] assignments of each expert on lower data-parallel ranks, or null (none)
  // extended step (kModeExt)
  const float* bias;           // [E] selection bias, or null (all zero)
  float bias_gamma;            // bias step
  float* bias_out;             // [E] updated bias (may alias bias), or null
  int masked_p;                // P over the picked experts only, divided by T*k
  const float* dgate;          // [T, k] upstream gradient of the gates, or null
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
  int32_t* tile_hist;          // [E][G_stride]: per-CTA counts
  int32_t* group_hist;         // [n_groups][E]: per-group counts (atomics; zero between launches)
  float* P_part;               // [E][G_stride]: per-CTA sums of p
  unsigned long long* pfix;    // [2][kMaxExperts]: a split step's sums of p in fixed point (zero between launches)
  int32_t* counts_ws;          // [E] counts when `counts` is not an output
  int G;                       // CTAs in the grid
  int n_groups;                // ceil(G / kGroupCtas)
  int G_stride;
  unsigned long long timeout_ns;
  unsigned barrier_extra;      // 0; 1 makes every grid barrier unreachable (timeout tests)
  unsigned long long* trace;   // [G][kTracePoints] phase timestamps (ns), or null
  // staging ring (staged variants)
  int rows_per_stage;
  int n_slots;
  int asg_cap;                 // assignments per CTA the shared-memory dispatch buffers hold (0: none)
  int rstat_cap;               // rows per CTA whose softmax statistics shared memory holds (0: none)
};

// Phase boundaries recorded in RouterParams::trace (lane 0 of the warp named).
enum : int {
  kTrStart = 0,        // warp 0: kernel entry
  kTrFirstStage,       // warp 0: first ring stage of the forward has landed
  kTrFwdRows,          // warp 0: its forward rows are done
  kTrFwdDone,          // warp 0: per-CTA counts and sums of p published
  kTrBarrier1,         // warp 0: first grid barrier passed
  kTrScanDone,         // warp 0: totals, this CTA's bases and the offsets are in shared memory
  kTrBarrier2,         // (not recorded)
  kTrBwdFirst,         // warp 0: first backward stage available
  kTrBwdRows,          // warp 0: its backward rows are done
  kTrDispatchDone,     // dispatch warp: dispatch (and CTA 0's E-sized outputs) done
  kTrJoined,           // warp 0: all warps joined
  kTrEnd,              // warp 0: kernel exit
  kTrRanked,           // dispatch warp: in-CTA dispatch ranks done
  kTrSmId,             // the SM the CTA runs on (an id, not a time)
  kTrFwdRowsAll,       // the last consumer warp's forward rows are done
  kTrBwdRowsAll,       // the last consumer warp's backward rows are done
  kTracePoints = 16
};

__device__ __forceinline__ void trace_point(const RouterParams& p, int point) {
  if (p.trace != nullptr && (threadIdx.x & 31) == 0) {
    if ((point == kTrDispatchDone || point == kTrRanked) ? threadIdx.x == kDispatchWarp * kWarp : threadIdx.x == 0) {
      p.trace[blockIdx.x * kTracePoints + point] = global_ns();
      if (point == kTrStart) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        p.trace[blockIdx.x * kTracePoints + kTrSmId] = smid;
      }
    }
  }
}

// Latest time over the calling warps (lane 0 of each) at `point`.
__device__ __forceinline__ void trace_last(const RouterParams& p, int point) {
  if (p.trace != nullptr && (threadIdx.x & 31) == 0) atomicMax(&p.trace[blockIdx.x * kTracePoints + point], global_ns());
}

struct BwdParams {
  const void* logits;
  long long T;
  int E;
  const float* f;
  float coef;                  // grad_scale * alpha * E / T
  float* dlogits;
};

// ---------------------------------------------------------------------------
// Shared-memory layout of the persistent kernel (byte offsets).
// ---------------------------------------------------------------------------
struct SmemLayout {
  unsigned red, hist, off, rank, w, bars, pick, rstat, asg, ring, total;
};

__host__ __device__ inline unsigned align_to(unsigned x, unsigned a) { return (x + a - 1) / a * a; }

// asg_cap: capacity of the two uint16 arrays (expert id and in-CTA rank of each
// of the CTA's assignments) that keep the dispatch in shared memory.
// rstat_cap: rows of (max, 1 / sum) kept from the forward for the backward.
// key_bytes: size of a top-k key (4 for bf16 logits, 8 for fp32).
__host__ __device__ inline SmemLayout router_smem_layout(int E, int key_bytes, int n_slots, int stage_bytes,
                                                         int asg_cap = 0, int rstat_cap = 0) {
  SmemLayout L;
  L.red = 0;                                                  // 128 ints
  L.hist = 512;                                               // E ints
  L.off = L.hist + 4u * E;                                    // E + 1 ints
  L.rank = L.off + 4u * (E + 1);                              // E ints
  L.w = align_to(L.rank + 4u * E, 16);                        // kConsumerWarps * E words
  L.bars = align_to(L.w + 4u * kConsumerWarps * E, 16);       // 2 * kMaxSlots mbarriers
  L.pick = L.bars + 16u * kMaxSlots;                          // kConsumerWarps * 64 keys
  L.rstat = L.pick + unsigned(key_bytes) * 64u * kConsumerWarps;   // rstat_cap float2
  L.asg = L.rstat + 8u * unsigned(rstat_cap);                 // 2 * asg_cap uint16
  L.ring = align_to(L.asg + 4u * unsigned(asg_cap), 128);
  L.total = L.ring + unsigned(n_slots) * unsigned(stage_bytes);
  return L;
}

// ---------------------------------------------------------------------------
// Vector loads / stores of VW elements.
// ---------------------------------------------------------------------------
template <int BYTES> struct VecT;
template <> struct VecT<2> { using T = uint16_t; };
template <> struct VecT<4> { using T = uint32_t; };
template <> struct VecT<8> { using T = uint2; };
template <> struct VecT<16> { using T = uint4; };

template <class Raw, int VW, bool GLOBAL>
__device__ __forceinline__ void load_vec(const Raw* src, Raw (&dst)[VW]) {
  constexpr int BYTES = int(sizeof(Raw)) * VW;
  if constexpr (BYTES <= 16) {
    using V = typename VecT<BYTES>::T;
    union { V v; Raw r[VW]; } u;
    if constexpr (GLOBAL) u.v = __ldg(reinterpret_cast<const V*>(src));
    else u.v = *reinterpret_cast<const V*>(src);
#pragma unroll
    for (int i = 0; i < VW; ++i) dst[i] = u.r[i];
  } else {
    constexpr int H = 16 / int(sizeof(Raw));
    static_assert(VW % H == 0, "vector width");
#pragma unroll
    for (int h = 0; h < VW / H; ++h) {
      union { uint4 v; Raw r[H]; } u;
      if constexpr (GLOBAL) u.v = __ldg(reinterpret_cast<const uint4*>(src + h * H));
      else u.v = *reinterpret_cast<const uint4*>(src + h * H);
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

template <int LPR, int VW>
__device__ __forceinline__ int col_of(int v, int l, int i) { return v * LPR * VW + l * VW + i; }
// The two disjoint bit fields of col_of (LPR and VW are powers of two): the
// lane's share, and the element's (a compile-time constant once unrolled).
template <int LPR, int VW>
__device__ __forceinline__ uint32_t col_lane_bits(int l) { return uint32_t(l * VW); }
template <int LPR, int VW>
__device__ __forceinline__ uint32_t col_elem_bits(int v, int i) { return uint32_t(v * LPR * VW + i); }

// Lane l's EPL elements of one row.  Columns past E read as -inf (their key is
// below every logit and their exp is 0, so the math needs no column checks);
// an invalid row reads as zeros.  `row` points at the row in global memory
// (GLOBAL) or in a ring stage.
template <class DT, int LPR, int VW, int NV, bool GLOBAL>
__device__ __forceinline__ void load_lane(const typename DT::Raw* row, int E, int l, bool valid,
                                          typename DT::Raw (&raw)[VW * NV]) {
  using Raw = typename DT::Raw;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int c0 = col_of<LPR, VW>(v, l, 0);
    Raw tmp[VW];
    if (valid && c0 < E) {   // E % VW == 0 for VW > 1: the whole vector is in the row
      load_vec<Raw, VW, GLOBAL>(row + c0, tmp);
    } else {
#pragma unroll
      for (int i = 0; i < VW; ++i) tmp[i] = valid ? DT::kNegInf : Raw(0);
    }
#pragma unroll
    for (int i = 0; i < VW; ++i) raw[v * VW + i] = tmp[i];
  }
}

// ---------------------------------------------------------------------------
// Forward of one row group: top-k on order-preserving keys, softmax against the
// row max, gates; idx/gate stores, pick counts into s_hist, p into pacc.
//
// Top-k.  Each lane keeps the two largest of its keys; k rounds take the group
// max of the lanes' heads, and the winning lane moves its second key up (a lane
// that has won twice is exhausted).  The rounds are exact unless some lane has
// a third key above the k-th pick; a count per lane detects that (rare) case
// and the row is then redone by exact_topk, which rescans.
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV, bool GLOBAL>
__device__ __forceinline__ void exact_topk(const typename DT::Raw* row, int E, int k, int l, bool valid,
                                        typename DT::Key* top_out, typename DT::Key* mine_out) {
  using Key = typename DT::Key;
  constexpr int EPL = VW * NV;
  typename DT::Raw raw[EPL];
  load_lane<DT, LPR, VW, NV, GLOBAL>(row, E, l, valid, raw);
  Key key[EPL];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; ++i)
      key[v * VW + i] = DT::key_from_bits(DT::canonical_zero(DT::bits(raw[v * VW + i])), col_lane_bits<LPR, VW>(l),
                                          col_elem_bits<LPR, VW>(v, i));
  Key prev = DT::kKeyMin, top = DT::kKeyMin, mine = DT::kKeyMin;
  for (int j = 0; j < k; ++j) {
    Key local = DT::kKeyMin;
#pragma unroll
    for (int i = 0; i < EPL; ++i) local = ((j == 0 || key[i] < prev) && key[i] > local) ? key[i] : local;
    const Key w = group_max_key<LPR>(local);
    if (j == 0) top = w;
    if (l == j) mine = w;
    prev = w;
  }
  *top_out = top;
  *mine_out = mine;
}

// Lane-local two largest keys of one row, as a pairwise tree (short dependency
// chains): merging sorted pairs (h1, l1) and (h2, l2) gives
// (max(h1, h2), max(min(h1, h2), l1, l2)).
__device__ __forceinline__ uint32_t max3_key(uint32_t a, uint32_t b, uint32_t c) { return __vimax3_u32(a, b, c); }
__device__ __forceinline__ long long max3_key(long long a, long long b, long long c) {
  const long long m = a > b ? a : b;
  return m > c ? m : c;
}

template <class Key, int EPL>
__device__ __forceinline__ void keys_top2(const Key (&key)[EPL], Key kmin, Key& m1, Key& m2) {
  if constexpr (EPL == 1) {
    m1 = key[0];
    m2 = kmin;
  } else {
    constexpr int N0 = (EPL + 1) / 2;
    Key hi[N0], lo[N0];
#pragma unroll
    for (int i = 0; i < EPL / 2; ++i) {
      const Key a = key[2 * i], b = key[2 * i + 1];
      hi[i] = a > b ? a : b;
      lo[i] = a < b ? a : b;
    }
    if constexpr (EPL & 1) {
      hi[N0 - 1] = key[EPL - 1];
      lo[N0 - 1] = kmin;
    }
#pragma unroll
    for (int n = N0; n > 1; n = (n + 1) / 2) {
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const Key a = hi[2 * i], b = hi[2 * i + 1];
        hi[i] = a > b ? a : b;
        lo[i] = max3_key(a < b ? a : b, lo[2 * i], lo[2 * i + 1]);
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

template <class DT, int LPR, int VW, int NV>
__device__ __forceinline__ void lane_top2(const typename DT::Raw (&raw)[VW * NV], int l, typename DT::Key& m1,
                                          typename DT::Key& m2) {
  using Key = typename DT::Key;
  constexpr int EPL = VW * NV;
  Key key[EPL];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; ++i)
      key[v * VW + i] = DT::key_from_bits(DT::bits(raw[v * VW + i]), col_lane_bits<LPR, VW>(l), col_elem_bits<LPR, VW>(v, i));
  keys_top2<Key, EPL>(key, DT::kKeyMin, m1, m2);
}

// Selection keys of the biased scores s = fp32(z) + b of lane l's elements
// ([P1] §4.3: the bias moves the choice of experts only): the fp32 keys of
// s (equal values tie, -0.0 with +0.0, and go to the lower column).  Columns
// past E hold -inf, whose score stays -inf whatever the bias there (zero).
template <class DT, int LPR, int VW, int NV>
__device__ __forceinline__ void biased_keys(const typename DT::Raw (&raw)[VW * NV], const float (&bl)[VW * NV], int l,
                                            long long (&key)[VW * NV]) {
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; ++i) {
      const float sc = __uint_as_float(DT::bits(raw[v * VW + i])) + bl[v * VW + i];
      key[v * VW + i] = Fp32::key_from_bits(__float_as_uint(sc), col_lane_bits<LPR, VW>(l), col_elem_bits<LPR, VW>(v, i));
    }
}

// Sum of x[0..N) in a fixed order: the pairs (x[2i], x[2i+1]) are added as
// packed fp32 pairs in a tree, then the pair's two halves, then the odd last
// element.
template <int N>
__device__ __forceinline__ float tree_sum(const float (&x)[N]) {
  if constexpr (N == 1) {
    return x[0];
  } else {
    constexpr int P = N / 2;
    float2 t[P];
#pragma unroll
    for (int i = 0; i < P; ++i) t[i] = make_float2(x[2 * i], x[2 * i + 1]);
#pragma unroll
    for (int n = P; n > 1; n = (n + 1) / 2) {
#pragma unroll
      for (int i = 0; i < n / 2; ++i) t[i] = add2(t[2 * i], t[2 * i + 1]);
      if (n & 1) t[n / 2] = t[n - 1];
    }
    float r = t[0].x + t[0].y;
    if constexpr (N & 1) r += x[N - 1];
    return r;
  }
}

// acc[i] += a[i] * b, two lanes at a time.
template <int N>
__device__ __forceinline__ void axpy2(float (&acc)[N], const float (&a)[N], float b) {
#pragma unroll
  for (int i = 0; i + 1 < N; i += 2) {
    const float2 r = fma2(make_float2(a[i], a[i + 1]), make_float2(b, b), make_float2(acc[i], acc[i + 1]));
    acc[i] = r.x;
    acc[i + 1] = r.y;
  }
  if constexpr (N & 1) acc[N - 1] = fmaf(a[N - 1], b, acc[N - 1]);
}

// Sum over the first min(LPR, 8) lanes of each row group (the owners of the k
// <= 8 picks; every other lane passes 0).
template <int LPR>
__device__ __forceinline__ float owners_sum(float x) {
#pragma unroll
  for (int off = 1; off < (LPR < 8 ? LPR : 8); off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Softmax numerators of lane l's share of a row against the row max m:
// e[i] = 2^(z_i * log2 e - mL) with mL = m * log2 e rounded once (one FFMA per
// element, ex2.approx, flush to zero).  The forward, both backward paths and
// the extension kernels use this one definition (and elem_exp for a single
// logit in fp32), so a row's p is the same bits wherever it is recomputed.
template <class DT, int LPR, int EPL>
__device__ __forceinline__ void row_exp(const typename DT::Raw (&raw)[EPL], float m, float (&e)[EPL]) {
  const float mL = m * kLog2e;
#pragma unroll
  for (int i = 0; i < EPL; ++i) e[i] = ex2_approx(fmaf(__uint_as_float(DT::bits(raw[i])), kLog2e, -mL));
}

// The numerator of one logit already in fp32, by the formula of row_exp.
__device__ __forceinline__ float elem_exp(float z, float m) { return ex2_approx(fmaf(z, kLog2e, -(m * kLog2e))); }

// d = a * b + c, clamped to [0, 1].
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---------------------------------------------------------------------------
// Fast top-k path for rows of 256 or more bf16 logits (32 lanes per row).
//
// Routing is skewed: most picks fall on a few experts.  Each CTA takes as
// candidates the 64 experts whose logits summed over the rows of its first
// ring stage are largest (an estimate of each expert's mean logit, which sets
// how often it lands in a row's top-k; choose_candidates).  For each later row
// every lane builds the keys of its two candidates' logits, k warp-wide rounds
// give the exact top-k among the 64, and a packed bf16 max over every other
// element of the row checks that none of them reaches the k-th pick's value.
// If one does (or ties it), the row is redone by the full path (lane_top2 and
// its rounds), so the result is exact for any input; the candidate set only
// decides how often the short path is enough.  A warp whose rows fail the
// check often stops trying.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The halves of w outside `keep` (0 there) replaced by -inf: (w & keep) | (~keep & -inf).
__device__ __forceinline__ uint32_t bf16x2_keep(uint32_t w, uint32_t keep) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xE2;" : "=r"(d) : "r"(w), "r"(keep), "r"(0xff80ff80u));
  return d;
}

// Order-preserving key of the bf16 value with fp32 bit pattern b (low half 0)
// in the column whose complement (0xffff - column) is inv: the key layout of
// Bf16::key_from_bits, for a column held in one register.
__device__ __forceinline__ uint32_t bf16_key_for(uint32_t b, uint32_t inv) {
  uint32_t s, k;
  asm("prmt.b32 %0, %1, %2, 0xBB54;" : "=r"(s) : "r"(b), "r"(inv));
  asm("lop3.b32 %0, %1, %2, %3, 0x16;" : "=r"(k) : "r"(b), "r"(s), "r"(0x80000000u));
  return k;
}

// Variants whose forward takes the fast path: bf16, 32 lanes per row, an even
// number of at most 16 elements per lane (E from 129 to 512).
template <class DT, int LPR, int VW, int NV>
constexpr bool kFastTopk = LPR == 32 && sizeof(typename DT::Raw) == 2 && VW % 2 == 0 && VW * NV <= 16;

// A consumer warp's share of the candidate set: one candidate per lane.
template <int NW>
struct FastTopk {
  int state;           // 0: candidates not chosen yet, 1: in use, 2: given up (warp-uniform)
  int tries, fails;    // rows tried and rows the check sent to the full path, since the last review
  uint32_t col0, col1; // this lane's two candidate columns
  uint32_t inv0, inv1; // 0xffff - col
  uint32_t keep[NW];   // per word of the lane's elements: 0xffff in each half whose column is not a candidate
};

// Adds column c of the rows [0, n) of a ring stage (bf16) into score[c]: the
// consumer warps split the columns between them, one per lane.
__device__ __forceinline__ void stage_column_sums(const uint16_t* st, int n, int E, int warp, float* score) {
  const int per = (E + kConsumerWarps - 1) / kConsumerWarps;    // <= 32 for E <= 576
  const int c = warp * per + (threadIdx.x & 31);
  if ((threadIdx.x & 31) < per && c < E) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int r = 0;
    for (; r + 4 <= n; r += 4)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] += __uint_as_float(uint32_t(st[(r + j) * E + c]) << 16);
    for (; r < n; ++r) acc[0] += __uint_as_float(uint32_t(st[r * E + c]) << 16);
    score[c] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  }
}

// Chooses the candidate set: the 64 columns with the largest scores (the
// columns' sums of the first stage's logits), by the upper 16 bits of their
// order-preserving images: those above the largest threshold th that at least
// 64 columns reach, then those at th in increasing column order.  Writes them
// as 16-bit pairs (lane l's two candidates in int l of the scratch), their
// membership bitmap, then the flag.  One warp; 64 < E <= 1024.
__device__ __forceinline__ void choose_candidates(const float* score, int E, int* s_red) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  constexpr int kCand = 2 * kWarp;
  auto key_of = [&](int e) -> uint32_t {
    const uint32_t b = __float_as_uint(score[e]);
    return ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) >> 16;
  };
  int lo_t = 0, hi_t = 0xffff;                   // #{key >= lo_t} >= 64 holds at lo_t = 0
  while (lo_t < hi_t) {
    const int mid = (lo_t + hi_t + 1) >> 1;
    int n = 0;
    for (int e = lane; e < E; e += kWarp) n += int(key_of(e)) >= mid ? 1 : 0;
    n = __reduce_add_sync(0xffffffffu, n);
    if (n >= kCand) lo_t = mid;
    else hi_t = mid - 1;
  }
  uint16_t* cand = reinterpret_cast<uint16_t*>(s_red + kRedCand);
  unsigned* bits = reinterpret_cast<unsigned*>(s_red + kRedCandBits);
  int base = 0;
  for (int pass = 0; pass < 2; ++pass) {         // above the threshold, then at it
    for (int e0 = 0; e0 < E && base < kCand; e0 += kWarp) {
      const int e = e0 + lane;
      const bool sel = e < E && (pass == 0 ? int(key_of(e)) > lo_t : int(key_of(e)) == lo_t);
      const unsigned b = __ballot_sync(0xffffffffu, sel);
      const int pos = base + __popc(b & lt);
      if (sel && pos < kCand) cand[pos] = uint16_t(e);
      base += __popc(b);
    }
  }
  bits[lane] = 0u;
  __syncwarp();
  for (int j = 0; j < 2; ++j) {
    const int c = cand[2 * lane + j];
    atomicOr(&bits[c >> 5], 1u << (c & 31));
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    *reinterpret_cast<volatile int*>(s_red + kRedCandReady) = 1;
  }
}

// Loads the candidate set into a consumer warp's FastTopk (after the flag).
template <int LPR, int VW, int NV>
__device__ __forceinline__ void fast_setup(FastTopk<VW * NV / 2>& fs, const int* s_red, int E, int l) {
  const unsigned* bits = reinterpret_cast<const unsigned*>(s_red + kRedCandBits);
  const uint16_t* cand = reinterpret_cast<const uint16_t*>(s_red + kRedCand);
  fs.col0 = cand[2 * (threadIdx.x & 31)];
  fs.col1 = cand[2 * (threadIdx.x & 31) + 1];
  fs.inv0 = 0xffffu - fs.col0;
  fs.inv1 = 0xffffu - fs.col1;
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; i += 2) {
      const int c = col_of<LPR, VW>(v, l, i);
      const bool in0 = c < E && ((bits[c >> 5] >> (c & 31)) & 1u);
      const bool in1 = c + 1 < E && ((bits[(c + 1) >> 5] >> ((c + 1) & 31)) & 1u);
      fs.keep[(v * VW + i) / 2] = (in0 ? 0u : 0x0000ffffu) | (in1 ? 0u : 0xffff0000u);
    }
  fs.state = 1;
  fs.tries = 0;
  fs.fails = 0;
}

// Lane l's EPL bf16 elements of one row (from a ring stage) as 32-bit words
// of two, columns past E as -inf, an invalid row as zeros.
template <int LPR, int VW, int NV>
__device__ __forceinline__ void load_lane_words(const uint16_t* row, int E, int l, bool valid,
                                                uint32_t (&wd)[VW * NV / 2]) {
  static_assert(VW == 2 || VW == 4 || VW == 8, "vector width");
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int c0 = col_of<LPR, VW>(v, l, 0);
    if (valid && c0 < E) {
      if constexpr (VW == 2) {
        wd[v] = *reinterpret_cast<const uint32_t*>(row + c0);
      } else if constexpr (VW == 4) {
        const uint2 q = *reinterpret_cast<const uint2*>(row + c0);
        wd[2 * v] = q.x;
        wd[2 * v + 1] = q.y;
      } else {
        const uint4 q = *reinterpret_cast<const uint4*>(row + c0);
        wd[4 * v] = q.x;
        wd[4 * v + 1] = q.y;
        wd[4 * v + 2] = q.z;
        wd[4 * v + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int h = 0; h < VW / 2; ++h) wd[v * VW / 2 + h] = valid ? 0xff80ff80u : 0u;
    }
  }
}

// The top key and lane l's pick (l < k) of one row.
template <class Key>
struct TopPick {
  Key top, mine;
};

// The full top-k of one row from a ring stage (32 lanes per row), out of
// line: lane_top2 and k rounds, then the exactness check of fwd_groups (a
// lane that spent both cached keys before the last round is counted exactly,
// and a row with a hidden key or a zero among its picks goes to exact_topk).
// It serves the rows of the fast path's first stage, the rows its check
// rejects and the warps that stopped trying it; kept out of line so that the
// fast path compiles lean.  Writes the picks to s_pick_row[0..k).
template <class DT, int VW, int NV>
__device__ __noinline__ TopPick<typename DT::Key> full_topk_row(const typename DT::Raw* row, int E, int k, int l,
                                                                 bool valid, typename DT::Key* s_pick_row) {
  using Key = typename DT::Key;
  constexpr int LPR = kWarp;
  constexpr int EPL = VW * NV;
  typename DT::Raw raw[EPL];
  load_lane<DT, LPR, VW, NV, false>(row, E, l, valid, raw);
  Key m1, m2;
  lane_top2<DT, LPR, VW, NV>(raw, l, m1, m2);
  const Key second = m2;
  __syncwarp();
  Key w = group_max_key<LPR>(m1);
  TopPick<Key> r;
  r.top = w;
  for (int j = 0;;) {
    s_pick_row[j] = w;
    const bool won = m1 == w;
    m1 = won ? m2 : m1;
    m2 = won ? DT::kKeyMin : m2;
    if (++j >= k) break;
    w = group_max_key<LPR>(m1);
  }
  __syncwarp();
  r.mine = l < k ? s_pick_row[l] : DT::kKeyMin;
  const bool early = EPL > 1 && m1 == DT::kKeyMin && second != w;
  bool redo = DT::kSplitsZero && __any_sync(0xffffffffu, valid && l < k && DT::is_zero(r.mine));
  if (!redo && __any_sync(0xffffffffu, early)) {
    int above = 0;
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i)
        above += DT::key_from_bits(DT::bits(raw[v * VW + i]), col_lane_bits<LPR, VW>(l), col_elem_bits<LPR, VW>(v, i)) > w
                     ? 1 : 0;
    redo = __any_sync(0xffffffffu, early && above > 2);
  }
  if (redo) exact_topk<DT, LPR, VW, NV, false>(row, E, k, l, valid, &r.top, &r.mine);
  return r;
}

// exact_topk of one row from a ring stage, out of line (a row of the fast
// path with a zero among its picks).
template <class DT, int VW, int NV>
__device__ __noinline__ TopPick<typename DT::Key> exact_topk_row(const typename DT::Raw* row, int E, int k, int l,
                                                                  bool valid) {
  TopPick<typename DT::Key> r;
  exact_topk<DT, kWarp, VW, NV, false>(row, E, k, l, valid, &r.top, &r.mine);
  return r;
}

// Shared-memory slots for one warp's picks: NR rows x (32 / LPR) groups x kMaxK.
constexpr int kPickSlotsPerWarp = 64;

// Forward of NR row groups of one warp at once (independent dependency chains
// interleave): top-k rounds, softmax against the row max (the first pick),
// gates; idx/gate stores, pick counts into s_hist, p into pacc.  s_pick is the
// warp's kPickSlotsPerWarp slots.  With s_aidx the expert ids also go to this
// CTA's shared-memory dispatch buffer (index a - a_base); with s_rstat each
// row's (max, 1 / sum) goes to s_rstat[t - r_base] for the backward.
template <class DT, int LPR, int VW, int NV, int NR, bool GLOBAL>
__device__ __forceinline__ void fwd_groups(const RouterParams& p, const typename DT::Raw* const (&row)[NR],
                                           const long long (&t)[NR], const bool (&valid)[NR], int l, int* s_hist,
                                           float (&pacc)[VW * NV], typename DT::Key* s_pick, uint16_t* s_aidx,
                                           long long a_base, float2* s_rstat, long long r_base) {
  using Raw = typename DT::Raw;
  using Key = typename DT::Key;
  constexpr int EPL = VW * NV;
  constexpr int GPW = kWarp / LPR;
  static_assert(NR * GPW * kMaxK <= kPickSlotsPerWarp, "pick slots");
  const int k = p.k;
  const int g = (threadIdx.x & 31) / LPR;

  Raw raw[NR][EPL];
  Key m1[NR], m2[NR], second[NR], top[NR], mine[NR], w[NR];
  float mx[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    load_lane<DT, LPR, VW, NV, GLOBAL>(row[r], p.E, l, valid[r], raw[r]);
    lane_top2<DT, LPR, VW, NV>(raw[r], l, m1[r], m2[r]);
    second[r] = m2[r];
  }
  // Round 0 gives the row max; the exponentials are issued before the other
  // rounds so that their latency hides behind them.  Round j's pick goes to
  // slot j of the row group; lane l takes pick l afterwards.
  float e[NR][EPL];
  __syncwarp();                                    // the previous rows' picks have been read
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    w[r] = group_max_key<LPR>(m1[r]);
    top[r] = w[r];
    s_pick[(r * GPW + g) * kMaxK] = w[r];
    const bool won = m1[r] == w[r];
    m1[r] = won ? m2[r] : m1[r];
    m2[r] = won ? DT::kKeyMin : m2[r];
    mx[r] = DT::key_value(top[r]);
    row_exp<DT, LPR, EPL>(raw[r], mx[r], e[r]);
  }
  {
    // Rounds 1 .. k - 1 in order: the switch enters the run of rounds k - 1
    // from its end, so no round tests k.
    Key* pk = s_pick + g * kMaxK + 1;
#define MOE_TOPK_ROUND                                                              \
    {                                                                               \
      _Pragma("unroll") for (int r = 0; r < NR; ++r) w[r] = group_max_key<LPR>(m1[r]); \
      _Pragma("unroll") for (int r = 0; r < NR; ++r) {                              \
        pk[r * GPW * kMaxK] = w[r];                                                 \
        const bool won = m1[r] == w[r];                                             \
        m1[r] = won ? m2[r] : m1[r];                                                \
        m2[r] = won ? DT::kKeyMin : m2[r];                                          \
      }                                                                             \
      ++pk;                                                                         \
    }
    static_assert(kMaxK == 8, "one case per k");
    switch (k) {
      case 8: MOE_TOPK_ROUND [[fallthrough]];
      case 7: MOE_TOPK_ROUND [[fallthrough]];
      case 6: MOE_TOPK_ROUND [[fallthrough]];
      case 5: MOE_TOPK_ROUND [[fallthrough]];
      case 4: MOE_TOPK_ROUND [[fallthrough]];
      case 3: MOE_TOPK_ROUND [[fallthrough]];
      case 2: MOE_TOPK_ROUND [[fallthrough]];
      default: break;
    }
#undef MOE_TOPK_ROUND
  }
  __syncwarp();
#pragma unroll
  for (int r = 0; r < NR; ++r) mine[r] = l < k ? s_pick[(r * GPW + g) * kMaxK + l] : DT::kKeyMin;

  // Only a lane that won twice before the last round can hide an unpicked
  // key above the k-th pick w (its cache is spent: m1 == kKeyMin, and its
  // second key was not the last pick); it does iff more than two of its keys
  // exceed w.  A count on the FMA pipe screens for that: every key above w
  // has e >= e(w) and adds 1, others add at most 1, so a lane whose count
  // stays at 2 hides nothing.  Rows that fail the screen get the exact count,
  // and exact_topk if needed.  With keys that rank -0.0 below +0.0, a row
  // whose picks include a zero is redone by exact_topk as well (the order of
  // equal logits decides it there).
  bool early[NR], check = false;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    early[r] = EPL > 1 && m1[r] == DT::kKeyMin && second[r] != w[r];
    check = check || early[r];
    if constexpr (DT::kSplitsZero) check = check || (valid[r] && l < k && DT::is_zero(mine[r]));
  }
  if (__any_sync(0xffffffffu, check)) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      bool redo = DT::kSplitsZero && __any_sync(0xffffffffu, valid[r] && l < k && DT::is_zero(mine[r]));
      if (!redo && __any_sync(0xffffffffu, early[r])) {
        const float ew = elem_exp(DT::key_value(w[r]), mx[r]);
        float est = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) est += fma_sat(e[r][i] - ew, 0x1p100f, 1.f);
        if (__any_sync(0xffffffffu, early[r] && est > 2.f)) {
          int above = 0;
#pragma unroll
          for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int i = 0; i < VW; ++i)
              above += DT::key_from_bits(DT::bits(raw[r][v * VW + i]), col_lane_bits<LPR, VW>(l),
                                         col_elem_bits<LPR, VW>(v, i)) > w[r] ? 1 : 0;
          redo = __any_sync(0xffffffffu, early[r] && above > 2);
        }
      }
      if (redo) exact_topk<DT, LPR, VW, NV, GLOBAL>(row[r], p.E, k, l, valid[r], &top[r], &mine[r]);
    }
  }

#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const float s = group_sum<LPR>(tree_sum(e[r]));
    const float inv_s = valid[r] ? rcp_approx(s) : 0.f;
    axpy2(pacc, e[r], inv_s);
    const bool owner = l < k;
    const float ej = owner ? elem_exp(DT::key_value(mine[r]), mx[r]) : 0.f;
    const float denom = p.renorm ? owners_sum<LPR>(ej) : s;
    if (valid[r] && owner) {
      const int col = DT::key_col(mine[r]);
      const long long a = t[r] * k + l;
      p.idx[a] = col;
      p.gate[a] = ej * rcp_approx(denom);
      atomicAdd(&s_hist[col], 1);
      if (s_aidx != nullptr) s_aidx[a - a_base] = uint16_t(col);
    }
    if (s_rstat != nullptr && valid[r] && l == 0) s_rstat[t[r] - r_base] = make_float2(mx[r], inv_s);
  }
}

// ---------------------------------------------------------------------------
// Forward of one row group of the extended step: top-k on the biased scores
// fp32(z) + b ([P1] §4.3; 64-bit keys, the rounds of fwd_groups, and for a lane
// that won twice the exact count of its keys above the k-th pick), softmax,
// gates and P from the unbiased z.  With masked P ([P2] §3.1) each pick adds
// its p into the warp's per-expert sums s_pm instead of pacc, in a fixed order.  bl: the bias of
// the lane's columns.
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV, bool GLOBAL>
__device__ __noinline__ long long exact_topk_ext(const typename DT::Raw* row, const float (&bl)[VW * NV], int E, int k,
                                                int l, bool valid) {
  constexpr int EPL = VW * NV;
  typename DT::Raw raw[EPL];
  load_lane<DT, LPR, VW, NV, GLOBAL>(row, E, l, valid, raw);
  long long key[EPL];
  biased_keys<DT, LPR, VW, NV>(raw, bl, l, key);
  long long prev = Fp32::kKeyMin, mine = Fp32::kKeyMin;
  for (int j = 0; j < k; ++j) {
    long long local = Fp32::kKeyMin;
#pragma unroll
    for (int i = 0; i < EPL; ++i) local = ((j == 0 || key[i] < prev) && key[i] > local) ? key[i] : local;
    const long long w = group_max_key<LPR>(local);
    if (l == j) mine = w;
    prev = w;
  }
  return mine;
}

// 32-bit selection key of a biased score s in column col < 1024: the
// order-preserving image of fp32 s (-0.0 taken as +0.0) with its low 10 bits
// replaced by 1023 - col, so equal images go to the lower column.  Scores whose
// images differ only in those 10 bits compare by column here: the row's picks
// are kept only when no such pair decides them (see fwd_groups_ext).
__device__ __forceinline__ uint32_t sel_key32(float sc, uint32_t col) {
  const uint32_t u = __float_as_uint(__fadd_rn(sc, 0.f));
  const uint32_t m = uint32_t(int(u) >> 31) | 0x80000000u;
  return ((u ^ m) | 0x3ffu) - col;
}
constexpr uint32_t kSelValueMask = 0xfffffc00u;

// Row max of finite-or-infinite floats: over 32 lanes by one warp reduction of
// the order-preserving images, else by shuffles.
template <int LPR>
__device__ __forceinline__ float group_max_img(float x) {
  if constexpr (LPR == 32) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t img = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    const uint32_t r = __reduce_max_sync(0xffffffffu, img);
    return __uint_as_float((r & 0x80000000u) ? (r & 0x7fffffffu) : ~r);
  } else {
    return group_max<LPR>(x);
  }
}

template <int LPR>
__device__ __forceinline__ int group_sum_int(int x) {
  if constexpr (LPR == 32) {
    return int(__reduce_add_sync(0xffffffffu, uint32_t(x)));
  } else {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
  }
}

template <class DT, int LPR, int VW, int NV, int NR, bool GLOBAL>
__device__ __forceinline__ void fwd_groups_ext(const RouterParams& p, const typename DT::Raw* const (&row)[NR],
                                               const long long (&t)[NR], const bool (&valid)[NR], int l, int* s_hist,
                                               float (&pacc)[VW * NV], uint32_t* s_pick, uint16_t* s_aidx,
                                               long long a_base, float2* s_rstat, long long r_base,
                                               const float (&bl)[VW * NV], float* s_pm) {
  using Raw = typename DT::Raw;
  constexpr int EPL = VW * NV;
  constexpr int GPW = kWarp / LPR;
  static_assert(NR * GPW * kMaxK <= kPickSlotsPerWarp, "pick slots");
  const int k = p.k, E = p.E;
  const int g = (threadIdx.x & 31) / LPR;
  const uint32_t lane_cols = col_lane_bits<LPR, VW>(l);

  Raw raw[NR][EPL];
  uint32_t key[NR][EPL], m1[NR], m2[NR], w[NR];
  float mx[NR], e[NR][EPL];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    load_lane<DT, LPR, VW, NV, GLOBAL>(row[r], E, l, valid[r], raw[r]);
    float m = -3.402823466e38f;
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VW; ++i) {
        const float z = __uint_as_float(DT::bits(raw[r][v * VW + i]));
        m = fmaxf(m, z);
        key[r][v * VW + i] = sel_key32(z + bl[v * VW + i], lane_cols + col_elem_bits<LPR, VW>(v, i));
      }
    keys_top2<uint32_t, EPL>(key[r], 0u, m1[r], m2[r]);
    mx[r] = group_max_img<LPR>(m);
    row_exp<DT, LPR, EPL>(raw[r], mx[r], e[r]);
  }
  __syncwarp();                                    // the previous rows' picks have been read
  for (int j = 0; j < k; ++j) {
#pragma unroll
    for (int r = 0; r < NR; ++r) w[r] = group_max_key<LPR>(m1[r]);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      s_pick[(r * GPW + g) * kMaxK + j] = w[r];
      const bool won = m1[r] == w[r];
      m1[r] = won ? m2[r] : m1[r];
      m2[r] = won ? 0u : m2[r];
    }
  }
  __syncwarp();
  // With bf16 logits and no bias the scores are bf16 values, whose images have
  // 16 zero low bits: the keys hold the whole scores and the rounds are exact
  // up to a lane that ran out of cached keys.  Otherwise the picks stand iff
  // exactly k elements have a value image at or above the k-th pick's (then
  // they are the picks: a lane that ran out of cached keys hid none, and no
  // other score shares the k-th one's image) and the picks' images are all
  // different (then their order is the scores' order).  Rows that fail are
  // redone on the full 64-bit keys.
  int col[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const uint32_t mine = l < k ? s_pick[(r * GPW + g) * kMaxK + l] : 0u;
    col[r] = int(1023u - (mine & 0x3ffu));
    const bool whole = sizeof(Raw) == 2 && p.bias == nullptr;
    const uint32_t thr = whole ? w[r] : (w[r] & kSelValueMask);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) cnt += key[r][i] >= thr ? 1 : 0;
    cnt = group_sum_int<LPR>(cnt);
    bool dup = false;
    if (!whole) {
      const uint32_t next = l + 1 < k ? s_pick[(r * GPW + g) * kMaxK + l + 1] : 0u;
      dup = l + 1 < k && (mine & kSelValueMask) == (next & kSelValueMask);
    }
    if (__any_sync(0xffffffffu, valid[r] && (cnt != k || dup))) {
      const long long m64 = exact_topk_ext<DT, LPR, VW, NV, GLOBAL>(row[r], bl, E, k, l, valid[r]);
      col[r] = l < k ? Fp32::key_col(m64) : 0;
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const float s = group_sum<LPR>(tree_sum(e[r]));
    const float inv_s = valid[r] ? rcp_approx(s) : 0.f;
    if (!p.masked_p) axpy2(pacc, e[r], inv_s);
    const bool owner = l < k;
    int c = 0;
    float ej = 0.f;
    if (owner) {
      c = min(max(col[r], 0), E - 1);
      Raw zr;
      if constexpr (GLOBAL) zr = __ldg(row[r] + c);
      else zr = row[r][c];
      ej = elem_exp(__uint_as_float(DT::bits(zr)), mx[r]);   // the unbiased numerator, as row_exp forms it
    }
    const float denom = p.renorm ? owners_sum<LPR>(ej) : s;
    if (valid[r] && owner) {
      const long long a = t[r] * k + l;
      p.idx[a] = c;
      p.gate[a] = ej * rcp_approx(denom);
      atomicAdd(&s_hist[c], 1);
      if (s_aidx != nullptr) s_aidx[a - a_base] = uint16_t(c);
    }
    // Masked P: the picks' p into the warp's sums, one row group after the
    // other (two groups' picks may share an expert), so the order of the
    // fp32 additions, and the result, is the same on every call.
    if (p.masked_p) {
#pragma unroll
      for (int gg = 0; gg < GPW; ++gg) {
        if (g == gg && valid[r] && owner) s_pm[c] += ej * inv_s;
        __syncwarp();
      }
    }
    if (s_rstat != nullptr && valid[r] && l == 0) s_rstat[t[r] - r_base] = make_float2(mx[r], inv_s);
  }
}

// Where a split step forms its renormalised gates: in the backward from 12
// elements per lane (E > 256: the forward is bound by instruction issue, the
// backward by memory, and the step at E = 384 is about 1 % faster), in the
// forward below (at E = 256, whose shorter backward carries k = 8, the
// backward's gates made the step 6 % slower).
template <int EPL>
constexpr bool kSplitGatesInBwd = EPL >= 12;

// The forward of the large-E bf16 variants (32 lanes per row, rows in a ring
// stage), in three parts: fast_topk_rows (the candidate path for K picks),
// full_topk_row (the full path, out of line) and row_tail (idx and, unless
// split, gate stores, pick counts, dispatch ids, row statistics).  A stage's rows
// take the candidate path one after the other and the ones it rejects are
// redone by the full path after the loop, so the per-row code has no rare
// branch in it.  SOFTMAX: the forward also forms the row's softmax (p into
// pacc, (max, 1 / sum) into s_rstat) and the gates; without it (the fused step
// with renormalised gates, whose backward forms the softmax sums and the
// gates) only the picks and the row max are kept.

// The candidate path for NR row groups: K rounds over the 64 candidates, then
// the check.  Returns (uniformly) whether every row passed; then top and
// mine hold each row's top key and lane l's pick.  A row whose picks include
// a zero does not pass (the order of equal logits decides it: the full path).
template <class DT, int VW, int NV, int NR, int K>
__device__ __forceinline__ bool fast_topk_rows(const typename DT::Raw* const (&row)[NR], const bool (&valid)[NR],
                                               int E, int l, typename DT::Key* s_pick, const FastTopk<(VW * NV) / 2>& fs,
                                               typename DT::Key (&top)[NR], typename DT::Key (&mine)[NR]) {
  using Key = typename DT::Key;
  constexpr int LPR = kWarp;
  constexpr int NW = VW * NV / 2;
  uint32_t wd[NR][NW];
  Key c1[NR], c2[NR], w[NR];                       // the lane's two candidate keys, larger first
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    load_lane_words<LPR, VW, NV>(row[r], E, l, valid[r], wd[r]);
    const uint32_t za = valid[r] ? uint32_t(row[r][fs.col0]) : 0u;
    const uint32_t zb = valid[r] ? uint32_t(row[r][fs.col1]) : 0u;
    const Key ka = bf16_key_for(za << 16, fs.inv0), kb = bf16_key_for(zb << 16, fs.inv1);
    c1[r] = ka > kb ? ka : kb;
    c2[r] = ka > kb ? kb : ka;
  }
  __syncwarp();                                    // the previous rows' picks have been read
#pragma unroll
  for (int j = 0; j < K; ++j) {
#pragma unroll
    for (int r = 0; r < NR; ++r) w[r] = group_max_key<LPR>(c1[r]);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      if (j == 0) top[r] = w[r];
      s_pick[r * kMaxK + j] = w[r];
      const bool won = c1[r] == w[r];
      c1[r] = won ? c2[r] : c1[r];
      c2[r] = won ? DT::kKeyMin : c2[r];
    }
  }
  // Every element outside the candidates must lie below the k-th pick's value.
  bool ok = true;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    uint32_t mw = bf16x2_keep(wd[r][0], fs.keep[0]);
#pragma unroll
    for (int j = 1; j < NW; ++j) mw = bf16x2_max(mw, bf16x2_keep(wd[r][j], fs.keep[j]));
    mw = bf16x2_max(mw, __byte_perm(mw, 0u, 0x1032));
    ok = ok && (!valid[r] || __uint_as_float(mw << 16) < DT::key_value(w[r]));
  }
  __syncwarp();
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    mine[r] = l < K ? s_pick[r * kMaxK + l] : DT::kKeyMin;
    ok = ok && !(valid[r] && l < K && DT::is_zero(mine[r]));
  }
  return __all_sync(0xffffffffu, ok);
}

// The rest of the forward of NR row groups once their picks are known.
template <class DT, int VW, int NV, int NR, bool SOFTMAX>
__device__ __forceinline__ void row_tail(const RouterParams& p, const typename DT::Raw* const (&row)[NR],
                                         const long long (&t)[NR], const bool (&valid)[NR], int l, int* s_hist,
                                         float (&pacc)[VW * NV], uint16_t* s_aidx, long long a_base, float2* s_rstat,
                                         long long r_base, const typename DT::Key (&top)[NR],
                                         const typename DT::Key (&mine)[NR]) {
  using Raw = typename DT::Raw;
  constexpr int LPR = kWarp;
  constexpr int EPL = VW * NV;
  const int k = p.k;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const float mx = DT::key_value(top[r]);
    const bool owner = l < k;
    float inv_s = 0.f;
    if constexpr (SOFTMAX) {
      const float ej = owner ? elem_exp(DT::key_value(mine[r]), mx) : 0.f;
      Raw raw[EPL];
      load_lane<DT, LPR, VW, NV, false>(row[r], p.E, l, valid[r], raw);
      float e[EPL];
      row_exp<DT, LPR, EPL>(raw, mx, e);
      const float s = group_sum<LPR>(tree_sum(e));
      inv_s = valid[r] ? rcp_approx(s) : 0.f;
      axpy2(pacc, e, inv_s);
      const float denom = p.renorm ? owners_sum<LPR>(ej) : s;
      if (valid[r] && owner) p.gate[t[r] * k + l] = ej * rcp_approx(denom);
    } else if constexpr (!kSplitGatesInBwd<EPL>) {
      const float ej = owner ? elem_exp(DT::key_value(mine[r]), mx) : 0.f;
      const float denom = owners_sum<LPR>(ej);
      if (valid[r] && owner) p.gate[t[r] * k + l] = ej * rcp_approx(denom);
    }
    // (otherwise a split step's renormalised gates are formed in its backward: split_gates)
    if (valid[r] && owner) {
      const int col = DT::key_col(mine[r]);
      const long long a = t[r] * k + l;
      p.idx[a] = col;
      atomicAdd(&s_hist[col], 1);
      if (s_aidx != nullptr) s_aidx[a - a_base] = uint16_t(col);
    }
    if (s_rstat != nullptr && valid[r] && l == 0) s_rstat[t[r] - r_base] = make_float2(mx, inv_s);
  }
}

// The full path for NR row groups, then the tail.
template <class DT, int VW, int NV, int NR, bool SOFTMAX>
__device__ __forceinline__ void slow_rows(const RouterParams& p, const typename DT::Raw* const (&row)[NR],
                                          const long long (&t)[NR], const bool (&valid)[NR], int l, int* s_hist,
                                          float (&pacc)[VW * NV], typename DT::Key* s_pick, uint16_t* s_aidx,
                                          long long a_base, float2* s_rstat, long long r_base) {
  typename DT::Key top[NR], mine[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const TopPick<typename DT::Key> tp = full_topk_row<DT, VW, NV>(row[r], p.E, p.k, l, valid[r], s_pick + r * kMaxK);
    top[r] = tp.top;
    mine[r] = tp.mine;
  }
  row_tail<DT, VW, NV, NR, SOFTMAX>(p, row, t, valid, l, s_hist, pacc, s_aidx, a_base, s_rstat, r_base, top, mine);
}

// The rest of a ring stage of a consumer warp on the candidate path with K
// picks: its row groups sg = sg0, sg0 + kConsumerWarps, ... take
// fast_topk_rows and the tail; the groups the check rejects are redone by the
// full path after the loop.  Returns the number of row groups tried; *failed
// gets the count rejected.
template <class DT, int VW, int NV, int NR, int K, bool SOFTMAX>
__device__ __forceinline__ int fast_stage(const RouterParams& p, const typename DT::Raw* st, int rows_here,
                                          long long t0, int sg0, int l, int* s_hist, float (&pacc)[VW * NV],
                                          typename DT::Key* s_pick, uint16_t* s_aidx, long long a_base,
                                          float2* s_rstat, long long r_base, const FastTopk<(VW * NV) / 2>& fs,
                                          int* failed_out) {
  using Raw = typename DT::Raw;
  const int E = p.E;
  unsigned failed = 0u;
  int n = 0;
  for (int sg = sg0; sg * NR < rows_here; sg += kConsumerWarps, ++n) {
    const Raw* rows[NR];
    long long ts[NR];
    bool valids[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const int ri = sg * NR + r;
      valids[r] = ri < rows_here;
      rows[r] = st + (valids[r] ? ri : 0) * E;
      ts[r] = t0 + ri;
    }
    typename DT::Key top[NR], mine[NR];
    if (fast_topk_rows<DT, VW, NV, NR, K>(rows, valids, E, l, s_pick, fs, top, mine))
      row_tail<DT, VW, NV, NR, SOFTMAX>(p, rows, ts, valids, l, s_hist, pacc, s_aidx, a_base, s_rstat, r_base, top, mine);
    else
      failed |= 1u << n;
  }
  *failed_out = __popc(failed);
  while (failed != 0u) {
    const int b = __ffs(failed) - 1;
    failed &= failed - 1u;
    const int sg = sg0 + b * kConsumerWarps;
    const Raw* rows[NR];
    long long ts[NR];
    bool valids[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const int ri = sg * NR + r;
      valids[r] = ri < rows_here;
      rows[r] = st + (valids[r] ? ri : 0) * E;
      ts[r] = t0 + ri;
    }
    slow_rows<DT, VW, NV, NR, SOFTMAX>(p, rows, ts, valids, l, s_hist, pacc, s_pick, s_aidx, a_base, s_rstat, r_base);
  }
  return n;
}

// A whole ring stage of a consumer warp in the large-E bf16 variants: the
// candidate path (k fixed per instantiation) while fs is in use, the full path
// otherwise.  A warp still waiting for the candidate set looks for it before
// each row group and switches as soon as it is published.
template <class DT, int VW, int NV, int NR, bool SOFTMAX>
__device__ __forceinline__ void fwd_stage_fast(const RouterParams& p, const typename DT::Raw* st, int rows_here,
                                               long long t0, int warp, int l, int* s_hist, float (&pacc)[VW * NV],
                                               typename DT::Key* s_pick, uint16_t* s_aidx, long long a_base,
                                               float2* s_rstat, long long r_base, FastTopk<(VW * NV) / 2>& fs,
                                               const int* s_red) {
  using Raw = typename DT::Raw;
  int sg = warp;
  for (; sg * NR < rows_here; sg += kConsumerWarps) {
    if (fs.state == 0 && *reinterpret_cast<const volatile int*>(s_red + kRedCandReady) != 0) {
      __threadfence_block();                       // the set itself after its flag
      fast_setup<kWarp, VW, NV>(fs, s_red, p.E, l);
    }
    if (fs.state == 1) break;
    const Raw* rows[NR];
    long long ts[NR];
    bool valids[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const int ri = sg * NR + r;
      valids[r] = ri < rows_here;
      rows[r] = st + (valids[r] ? ri : 0) * p.E;
      ts[r] = t0 + ri;
    }
    slow_rows<DT, VW, NV, NR, SOFTMAX>(p, rows, ts, valids, l, s_hist, pacc, s_pick, s_aidx, a_base, s_rstat, r_base);
  }
  if (fs.state == 1 && sg * NR < rows_here) {
    int n = 0, failed = 0;
#define MOE_FAST_STAGE(K)                                                                                        \
    n = fast_stage<DT, VW, NV, NR, K, SOFTMAX>(p, st, rows_here, t0, sg, l, s_hist, pacc, s_pick, s_aidx, a_base, \
                                               s_rstat, r_base, fs, &failed)
    switch (p.k) {
      case 1: MOE_FAST_STAGE(1); break;
      case 2: MOE_FAST_STAGE(2); break;
      case 3: MOE_FAST_STAGE(3); break;
      case 4: MOE_FAST_STAGE(4); break;
      case 5: MOE_FAST_STAGE(5); break;
      case 6: MOE_FAST_STAGE(6); break;
      case 7: MOE_FAST_STAGE(7); break;
      default: MOE_FAST_STAGE(8); break;
    }
#undef MOE_FAST_STAGE
    fs.tries += n;
    fs.fails += failed;
  }
}

// ---------------------------------------------------------------------------
// Backward of one row group:
//   dlogits[t,j] = coef * p[t,j] * (f[j] - sum_i p[t,i] f[i])
// With F = coef * f (held per lane), p = e / s and w = (1/s)^2 * sum_i e_i F_i:
//   dlogits[t,j] = e_j * ((1/s) * F_j - w).
// The row max mx and inv_s come from the forward (bwd_row_stats otherwise).
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV>
__device__ __forceinline__ void bwd_row_stats(const typename DT::Raw (&raw)[VW * NV], float& mx, float& inv_s) {
  constexpr int EPL = VW * NV;
  float m = -3.402823466e38f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) m = fmaxf(m, __uint_as_float(DT::bits(raw[i])));
  mx = group_max<LPR>(m);
  float e[EPL];
  row_exp<DT, LPR, EPL>(raw, mx, e);
  inv_s = rcp_approx(group_sum<LPR>(tree_sum(e)));
}

template <class DT, int LPR, int VW, int NV>
__device__ __forceinline__ void bwd_group(const typename DT::Raw (&raw)[VW * NV], const float (&Fr)[VW * NV], long long t,
                                          bool valid, int l, int E, float mx, float inv_s, float* dlogits) {
  constexpr int EPL = VW * NV;
  float e[EPL];
  row_exp<DT, LPR, EPL>(raw, mx, e);
  float dot[EPL];
#pragma unroll
  for (int i = 0; i + 1 < EPL; i += 2) {
    const float2 q = mul2(make_float2(e[i], e[i + 1]), make_float2(Fr[i], Fr[i + 1]));
    dot[i] = q.x;
    dot[i + 1] = q.y;
  }
  if constexpr (EPL & 1) dot[EPL - 1] = e[EPL - 1] * Fr[EPL - 1];
  const float w = inv_s * (inv_s * group_sum<LPR>(tree_sum(dot)));
  if (valid) {
    float* out = dlogits + t * (long long)E;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int c0 = col_of<LPR, VW>(v, l, 0);
      if (c0 < E) {
        float d[VW];
        if constexpr (VW % 2 == 0) {
#pragma unroll
          for (int i = 0; i < VW; i += 2) {
            const int j = v * VW + i;
            const float2 h = fma2(make_float2(inv_s, inv_s), make_float2(Fr[j], Fr[j + 1]), make_float2(-w, -w));
            const float2 q = mul2(make_float2(e[j], e[j + 1]), h);
            d[i] = q.x;
            d[i + 1] = q.y;
          }
        } else {
#pragma unroll
          for (int i = 0; i < VW; ++i) d[i] = e[v * VW + i] * fmaf(inv_s, Fr[v * VW + i], -w);
        }
        store_vec_f32<VW>(out + c0, d);
      }
    }
  }
}

// Backward of one row group in a split step: the softmax sum comes here, not
// from the forward.  e, s = sum e and sum e * F are formed in one pass (the
// same arithmetic and order as bwd_row_stats and bwd_group, so dlogits is the
// same bits as the separate backward's); p = e / s is added into pacc.
template <class DT, int LPR, int VW, int NV>
__device__ __forceinline__ void bwd_group_split(const typename DT::Raw (&raw)[VW * NV], const float (&Fr)[VW * NV],
                                                long long t, bool valid, int l, int E, float mx, float (&pacc)[VW * NV],
                                                float* dlogits) {
  constexpr int EPL = VW * NV;
  float e[EPL];
  row_exp<DT, LPR, EPL>(raw, mx, e);
  float dot[EPL];
#pragma unroll
  for (int i = 0; i + 1 < EPL; i += 2) {
    const float2 q = mul2(make_float2(e[i], e[i + 1]), make_float2(Fr[i], Fr[i + 1]));
    dot[i] = q.x;
    dot[i + 1] = q.y;
  }
  if constexpr (EPL & 1) dot[EPL - 1] = e[EPL - 1] * Fr[EPL - 1];
  float sum = tree_sum(e), sdot = tree_sum(dot);
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) {
    sum += __shfl_xor_sync(0xffffffffu, sum, off);
    sdot += __shfl_xor_sync(0xffffffffu, sdot, off);
  }
  const float inv_s = rcp_approx(sum);
  if (valid) axpy2(pacc, e, inv_s);
  const float w = inv_s * (inv_s * sdot);
  if (valid) {
    float* out = dlogits + t * (long long)E;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int c0 = col_of<LPR, VW>(v, l, 0);
      if (c0 < E) {
        float d[VW];
#pragma unroll
        for (int i = 0; i < VW; i += 2) {
          const int j = v * VW + i;
          const float2 h = fma2(make_float2(inv_s, inv_s), make_float2(Fr[j], Fr[j + 1]), make_float2(-w, -w));
          const float2 q = mul2(make_float2(e[j], e[j + 1]), h);
          d[i] = q.x;
          d[i + 1] = q.y;
        }
        store_vec_f32<VW>(out + c0, d);
      }
    }
  }
}

// Lane l's upstream gradient of gate l of row t (zero off the picks' lanes,
// past the batch, or without dgate).
__device__ __forceinline__ float dgate_of(const RouterParams& p, long long t, int l, bool valid) {
  return valid && l < p.k && p.dgate != nullptr ? __ldg(p.dgate + t * p.k + l) : 0.f;
}

// The extended backward's gate terms of a warp's rows of one ring stage, ahead
// of the rows (pre-pass): 8 lanes per row and 4 rows at a time, lane j of a
// row taking pick j (its column, its numerator from the row, its upstream
// gradient: the loads of 4 rows in flight together), and gp_j = p_j gamma_j as
// bwd_group_ext forms it (renormalised gates: the differences dgate_j -
// dgate_m over the row's 8-lane segment).  gp_out[slot * kMaxK + j], slot =
// n * RPW + g for the warp's n-th row group of the stage, its group g.  Needs
// the forward's row statistics in shared memory.
template <class DT, int LPR>
__device__ __forceinline__ void ext_gate_prepass(const RouterParams& p, const typename DT::Raw* st, long long t0,
                                                 int rs0, int rows_here, int warp, int n_rows, const float2* s_rstat,
                                                 const uint16_t* s_aidx, long long a_base, float coef_m,
                                                 const float* s_f, float* gp_out) {
  constexpr int RPW = kWarp / LPR;
  const int lane = threadIdx.x & 31;
  const int k = p.k, E = p.E;
  for (int base = 0; base < n_rows; base += kWarp / kMaxK) {
    const int slot = base + lane / kMaxK, j = lane % kMaxK;
    const int n = slot / RPW, g = slot % RPW;
    const int ri = (warp + n * kConsumerWarps) * RPW + g;
    const bool owner = slot < n_rows && ri < rows_here && j < k;
    float ec = 0.f, dg = 0.f, inv_s = 0.f;
    int col = 0;
    if (owner) {
      const long long a = (t0 + ri) * k + j;
      col = s_aidx != nullptr ? int(s_aidx[a - a_base]) : __ldcg(p.idx + a);
      col = min(max(col, 0), E - 1);
      const float2 rs = s_rstat[rs0 + ri];
      inv_s = rs.y;
      ec = elem_exp(__uint_as_float(DT::bits(st[ri * E + col])), rs.x);
      if (p.dgate != nullptr) dg = __ldg(p.dgate + a);
    }
    float gp = 0.f;
    if (p.dgate != nullptr) {
      if (p.renorm) {
        float Se = ec, acc = 0.f;
#pragma unroll
        for (int o = 1; o < kMaxK; ++o) {
          const float ep = __shfl_xor_sync(0xffffffffu, ec, o);
          const float dp = __shfl_xor_sync(0xffffffffu, dg, o);
          Se += ep;
          acc = fmaf(ep, dg - dp, acc);
        }
        const float inv_Se = rcp_approx(Se);
        gp = owner ? ec * (acc * inv_Se) * inv_Se : 0.f;
      } else {
        gp = owner ? ec * inv_s * dg : 0.f;
      }
    }
    if (p.masked_p && owner) gp = fmaf(ec * inv_s, coef_m * s_f[col], gp);
    if (slot < n_rows) gp_out[slot * kMaxK + j] = gp;
  }
  __syncwarp();
}

// Backward of one row group of the extended step: dlogits = p * (dp - sum p dp)
// for L = sum_j dgate_j * gate_j + grad_scale * L_aux (picks and f fixed).  Fr
// holds coef * f on the lane's columns (zero with masked P).  Lane j < k of the
// group takes pick j: its column (the forward's idx), its numerator ec (the
// bits row_exp gives it) and gp = p_j * gamma_j, gamma_j its extra dL/dp: the
// gate term (renormalised: (dgate_j - G) / sum_m p_m with G = sum_m dgate_m
// gate_m, so gp = gate_j (dgate_j - G), formed from the differences dgate_j -
// dgate_m; plain: dgate_j) and with masked P the
// aux term coef_m * f_j.  Every lane stores p * (F - S) with S = sum p F +
// sum gp; then, after a warp sync, lane j stores its pick's element again with
// gp added.  dg_in: lane j's upstream
// gradient of gate j of this row (loaded ahead by the caller).
template <class DT, int LPR, int VW, int NV, bool GLOBAL>
__device__ __forceinline__ void bwd_group_ext(const RouterParams& p, const typename DT::Raw (&raw)[VW * NV],
                                              const typename DT::Raw* row, const float (&Fr)[VW * NV], long long t,
                                              bool valid, int l, int E, float mx, float inv_s, float coef_f,
                                              float coef_m, const float* s_f, const uint16_t* s_aidx, long long a_base,
                                              float dg_in, const float* gp_pre, int slot) {
  constexpr int EPL = VW * NV;
  const int k = p.k;
  // the pick's loads first: their latency hides behind the row's arithmetic
  const bool owner = valid && l < k;
  int col = 0;
  const float dg = owner ? dg_in : 0.f;
  typename DT::Raw zr = DT::kNegInf;
  if (owner) {
    const long long a = t * k + l;
    col = s_aidx != nullptr ? int(s_aidx[a - a_base]) : __ldcg(p.idx + a);
    col = min(max(col, 0), E - 1);
    if constexpr (GLOBAL) zr = __ldg(row + col);
    else zr = row[col];
  }
  float e[EPL];
  row_exp<DT, LPR, EPL>(raw, mx, e);
  float dot[EPL];
#pragma unroll
  for (int i = 0; i + 1 < EPL; i += 2) {
    const float2 q = mul2(make_float2(e[i], e[i + 1]), make_float2(Fr[i], Fr[i + 1]));
    dot[i] = q.x;
    dot[i + 1] = q.y;
  }
  if constexpr (EPL & 1) dot[EPL - 1] = e[EPL - 1] * Fr[EPL - 1];
  const float wa = inv_s * (inv_s * group_sum<LPR>(tree_sum(dot)));
  const float ec = owner ? elem_exp(__uint_as_float(DT::bits(zr)), mx) : 0.f;
  float gp = 0.f;
  if (gp_pre != nullptr) {
    gp = owner ? gp_pre[slot * kMaxK + l] : 0.f;   // formed ahead by ext_gate_prepass
  } else if (p.dgate != nullptr) {
    if (p.renorm) {
      // gate_j (dgate_j - G) as e_j sum_m e_m (dgate_j - dgate_m) / Se^2: the
      // differences term by term, which do not cancel as dgate_j - G can
      const int base = (threadIdx.x & 31) - l;    // lane 0 of the group
      float Se = 0.f, acc = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          const float ej = __shfl_sync(0xffffffffu, ec, base + j);
          const float dj = __shfl_sync(0xffffffffu, dg, base + j);
          Se += ej;
          acc = fmaf(ej, dg - dj, acc);
        }
      }
      const float inv_Se = rcp_approx(Se);
      gp = owner ? ec * (acc * inv_Se) * inv_Se : 0.f;
    } else {
      gp = owner ? ec * inv_s * dg : 0.f;
    }
  }
  if (gp_pre == nullptr && p.masked_p && owner) gp = fmaf(ec * inv_s, coef_m * s_f[col], gp);
  // S = sum p F + sum gp.  With renormalised gates and no masked term the gate
  // part sums to zero over the picks (sum_j gate_j (dgate_j - G) = 0), so it
  // is left out rather than added as rounding noise.
  const bool gate_sum = p.masked_p || (p.dgate != nullptr && !p.renorm);
  const float w = gate_sum ? fmaf(inv_s, group_sum<LPR>(gp), wa) : wa;
  if (valid) {
    float* out = p.dlogits + t * (long long)E;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int c0 = col_of<LPR, VW>(v, l, 0);
      if (c0 < E) {
        float d[VW];
        if constexpr (VW % 2 == 0) {
#pragma unroll
          for (int i = 0; i < VW; i += 2) {
            const int j = v * VW + i;
            const float2 h = fma2(make_float2(inv_s, inv_s), make_float2(Fr[j], Fr[j + 1]), make_float2(-w, -w));
            const float2 q = mul2(make_float2(e[j], e[j + 1]), h);
            d[i] = q.x;
            d[i + 1] = q.y;
          }
        } else {
#pragma unroll
          for (int i = 0; i < VW; ++i) d[i] = e[v * VW + i] * fmaf(inv_s, Fr[v * VW + i], -w);
        }
        store_vec_f32<VW>(out + c0, d);
      }
    }
  }
  __syncwarp();                                    // the pick's element above is stored first
  if (owner) {
    const float F = coef_f * s_f[col];
    __stcs(p.dlogits + t * (long long)E + col, fmaf(ec, fmaf(inv_s, F, -w), gp));
  }
}

// A split step's renormalised gates of one row, in its backward (the forward
// is bound by instruction issue, the backward by memory): lane j < k takes
// pick j from the dispatch ids in shared memory (or the idx the forward
// wrote), its logit from the row, and forms gate_j = e_j / sum_m e_m with the
// arithmetic the forward would have used (the same row max, elem_exp).
template <class DT, int LPR>
__device__ __forceinline__ void split_gates(const RouterParams& p, const typename DT::Raw* row, long long t, bool valid,
                                            int l, float mx, const uint16_t* s_aidx, long long a_base) {
  const int k = p.k;
  const bool owner = valid && l < k;
  float ej = 0.f;
  if (owner) {
    const long long a = t * k + l;
    int col = s_aidx != nullptr ? int(s_aidx[a - a_base]) : __ldcg(p.idx + a);
    col = min(max(col, 0), p.E - 1);
    ej = elem_exp(__uint_as_float(DT::bits(row[col])), mx);
  }
  const float denom = owners_sum<LPR>(ej);
  if (owner) p.gate[t * k + l] = ej * rcp_approx(denom);
}

// A CTA's sum of p of one expert (x >= 0) into the fixed-point totals: its
// value split at 2^-20 and 2^-64 into two 64-bit integers, so the totals are
// exact whatever the order of the atomics.
__device__ __forceinline__ void pfix_add(unsigned long long* hi_acc, unsigned long long* lo_acc, float x) {
  const double q = double(x) * 0x1p20;                 // x < 2^31: q < 2^51
  const double hi = floor(q);
  const unsigned long long lo = (unsigned long long)((q - hi) * 0x1p44);   // exact for x >= 2^-41
  if (hi != 0.0) atomicAdd(hi_acc, (unsigned long long)hi);
  if (lo != 0ull) atomicAdd(lo_acc, lo);
}

// The value of a fixed-point total.
__device__ __forceinline__ double pfix_value(unsigned long long hi, unsigned long long lo) {
  return double(hi) * 0x1p-20 + double(lo) * 0x1p-64;
}

// Lane l's values of coef * f (zero past E) from a shared-memory copy of f.
template <int LPR, int VW, int NV>
__device__ __forceinline__ void load_f(const float* s_f, int E, int l, float coef, float (&Fr)[VW * NV]) {
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < VW; ++i) {
      const int c = col_of<LPR, VW>(v, l, i);
      Fr[v * VW + i] = c < E ? coef * s_f[c] : 0.f;
    }
}

__device__ __forceinline__ void sync_main() {
  asm volatile("bar.sync %0, %1;" :: "n"(kBarMain), "n"(kMainThreads) : "memory");
}

// ---------------------------------------------------------------------------
// The sum over the G CTAs of one expert's per-CTA sums of p, by one warp, in a
// fixed order: lane l adds the consecutive CTAs [l * per, (l + 1) * per), then
// the lanes are added pairwise.
// ---------------------------------------------------------------------------
constexpr int kColPerLane = 32;   // kGridMax / 32
__device__ __forceinline__ float warp_column_sum_f(const float* col, int G) {
  static_assert(kGridMax <= kWarp * kColPerLane, "column width");
  const int lane = threadIdx.x & 31;
  const int per = (G + kWarp - 1) / kWarp;
  const int c0 = min(lane * per, G), c1 = min(c0 + per, G);
  float v[kColPerLane];
#pragma unroll
  for (int i = 0; i < kColPerLane; ++i) v[i] = c0 + i < c1 ? __ldcg(col + c0 + i) : 0.f;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kColPerLane; ++i) s += v[i];
  return warp_sum_f(s);
}

// Per-expert totals and this CTA's dispatch bases (the counts of the CTAs
// before it), by the main group: S consecutive lanes share an expert (S the
// largest power of two up to 32 with E * S <= kMainThreads), each reads its
// share of the expert's group sums and of the counts of this CTA's
// predecessors within its group (all loads in flight together), and the S
// partial sums are added by shuffles.  Writes total[e] and base[e] for every
// expert; the caller syncs the main group.
__device__ __forceinline__ void totals_and_bases(const RouterParams& p, int cta, int* total, int* base) {
  const int E = p.E, tid = threadIdx.x;
  const int grp = cta / kGroupCtas;
  const int n_pre = cta - grp * kGroupCtas;            // predecessors within the group
  const int n_items = p.n_groups + n_pre;              // per expert: group sums, then predecessors
  int S = 32;
  while (S > 1 && E * S > kMainThreads) S >>= 1;
  const int s = tid & (S - 1);
  constexpr int kB = 16;                               // loads per lane in flight together
  static_assert(kMainThreads % kWarp == 0, "whole warps");
  const int per_trip = kMainThreads / S;               // experts per trip (S divides kMainThreads)
  const int trips = (E + per_trip - 1) / per_trip;     // the same for every thread: the shuffles need whole warps
  for (int r = 0; r < trips; ++r) {
    const int e = r * per_trip + tid / S;
    const bool on = e < E;
    int tot = 0, pre = 0;
    for (int i0 = s; i0 < n_items; i0 += kB * S) {
      int v[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int i = i0 + j * S;
        v[j] = 0;
        if (on && i < p.n_groups) v[j] = __ldcg(p.group_hist + (size_t)i * E + e);
        else if (on && i < n_items) v[j] = __ldcg(p.tile_hist + (size_t)e * p.G_stride + grp * kGroupCtas + (i - p.n_groups));
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int i = i0 + j * S;
        if (i < p.n_groups) {
          tot += v[j];
          pre += i < grp ? v[j] : 0;
        } else {
          pre += v[j];
        }
      }
    }
    for (int o = 1; o < S; o <<= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      pre += __shfl_xor_sync(0xffffffffu, pre, o);
    }
    if (on && s == 0) {
      total[e] = tot;
      base[e] = pre;
    }
  }
}

// ---------------------------------------------------------------------------
// Dispatch.  The stable rank of assignment a = t*k + j among the assignments
// to its expert e is  (count of e in the CTAs before this one)  +  (count of e
// among this CTA's assignments before a).  A warp walks a run of assignments
// in order, 32 at a time: lanes holding the same expert are found with one
// match.any, and a per-expert running count in shared memory gives the rank
// within the run.  With the rows streamed through the ring this
// runs during the forward, a stage behind the consumer warps, and parks the
// in-CTA ranks in slot[]; after the global prefix is known a sync-free pass
// turns them into final ranks and writes perm and slot.
// ---------------------------------------------------------------------------
constexpr int kDispChunks = 8;

// How idx is read: a read-only input, data this CTA is writing during the
// forward (volatile loads, coherent within the SM), or data published before a
// grid barrier (L2 loads).
enum : int { kLoadInput = 0, kLoadOwn = 1, kLoadPublished = 2 };

// In-CTA ranks of assignments [a_lo, a_hi), written to out[a].
template <int LOAD>
__device__ __forceinline__ void local_ranks(const int32_t* idx_src, long long a_lo, long long a_hi, int E, int* rank,
                                            int32_t* out) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (long long base = a_lo; base < a_hi; base += kDispChunks * kWarp) {
    int e_[kDispChunks], r_[kDispChunks];
#pragma unroll
    for (int j = 0; j < kDispChunks; ++j) {
      const long long a = base + j * kWarp + lane;
      int v = 0;
      if (a < a_hi) {
        if constexpr (LOAD == kLoadOwn) v = *reinterpret_cast<const volatile int32_t*>(idx_src + a);
        else if constexpr (LOAD == kLoadPublished) v = __ldcg(idx_src + a);
        else v = __ldg(idx_src + a);
      }
      e_[j] = min(max(v, 0), E - 1);
    }
#pragma unroll
    for (int j = 0; j < kDispChunks; ++j) {
      r_[j] = 0;
      if (base + j * kWarp >= a_hi) continue;             // warp-uniform
      const bool act = base + j * kWarp + lane < a_hi;
      const int e = e_[j];
      // lanes holding the same expert (an inactive lane matches only itself)
      const unsigned peers = __match_any_sync(0xffffffffu, act ? e : E + lane);
      const int lower = __popc(peers & lt);
      r_[j] = act ? rank[e] + lower : 0;
      __syncwarp();
      if (act && lower == 0) rank[e] += __popc(peers);
      __syncwarp();
    }
#pragma unroll
    for (int j = 0; j < kDispChunks; ++j) {
      const long long a = base + j * kWarp + lane;
      if (a < a_hi) out[a] = r_[j];
    }
  }
}

// Slot of an assignment with rank r among this batch's assignments to expert
// e: its position r + cap_base[e] in the expert's buffer when that is below
// the capacity, else -1 (dropped).  cap_base (the expert's assignments on the
// lower data-parallel ranks) is null for a batch on one rank.
__device__ __forceinline__ int slot_of(const RouterParams& p, int e, int r) {
  const int g = p.cap_base != nullptr ? r + __ldg(p.cap_base + e) : r;
  return g < p.C ? g : -1;
}

// Final ranks from the parked in-CTA ranks: r = base[e] + local; perm and slot.
__device__ __forceinline__ void dispatch_fixup(const RouterParams& p, const int32_t* idx_src, long long a0, long long a1,
                                               const int* off, const int* base) {
  const int lane = threadIdx.x & 31;
  const int E = p.E;
  for (long long b = a0; b < a1; b += 4 * kWarp) {
    int e_[4], l_[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long a = b + j * kWarp + lane;
      e_[j] = a < a1 ? min(max(__ldcg(idx_src + a), 0), E - 1) : 0;
      l_[j] = a < a1 ? __ldcg(p.slot + a) : 0;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long a = b + j * kWarp + lane;
      const int e = e_[j];
      const int r = base[e] + l_[j];
      if (a < a1 && r >= 0 && r < off[e + 1] - off[e]) {   // always true for consistent ranks
        p.perm[off[e] + r] = int(a);
        p.slot[a] = slot_of(p, e, r);
      }
    }
  }
}

// In-CTA ranks from the shared-memory copy of this CTA's expert ids: for local
// assignment indices [lo, hi), rank[lo..hi) = rank among this CTA's assignments
// to the same expert.
__device__ __forceinline__ void local_ranks_smem(const uint16_t* aidx, int lo, int hi, int* rank, uint16_t* out) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = lo; base < hi; base += kWarp) {
    const int a = base + lane;
    const bool act = a < hi;
    const int e = act ? aidx[a] : 0;
    // lanes holding the same expert (an inactive lane matches only itself)
    const unsigned peers = __match_any_sync(0xffffffffu, act ? e : kCtrlNoExpert + lane);
    const int lower = __popc(peers & lt);
    const int r = act ? rank[e] + lower : 0;
    __syncwarp();
    if (act && lower == 0) rank[e] += __popc(peers);
    __syncwarp();
    if (act) out[a] = uint16_t(r);
  }
}

// Final positions from the shared-memory expert ids and in-CTA ranks.
__device__ __forceinline__ void dispatch_fixup_smem(const RouterParams& p, long long a0, int n, const uint16_t* aidx,
                                                    const uint16_t* arank, const int* off, const int* base) {
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < n; i += kWarp) {
    const int e = aidx[i];
    const int r = base[e] + arank[i];
    const long long a = a0 + i;
    if (r >= 0 && r < off[e + 1] - off[e]) {                // always true for consistent ranks
      p.perm[off[e] + r] = int(a);
      p.slot[a] = slot_of(p, e, r);
    }
  }
}

// Final ranks directly (rank[e] starts at the CTA's prefix), for the variants
// that read rows straight from global memory: used after the global prefix.
__device__ __forceinline__ void dispatch_direct(const RouterParams& p, const int32_t* idx_src, long long a0, long long a1,
                                                const int* off, int* rank) {
  const int E = p.E;
  const int lane = threadIdx.x & 31;
  local_ranks<kLoadPublished>(idx_src, a0, a1, E, rank, p.slot);   // slot[a] = final rank
  __syncwarp();
  for (long long a = a0 + lane; a < a1; a += kWarp) {
    const int e = min(max(__ldcg(idx_src + a), 0), E - 1);
    const int r = p.slot[a];
    if (r >= 0 && r < off[e + 1] - off[e]) {                // always true for consistent ranks
      p.perm[off[e] + r] = int(a);
      p.slot[a] = slot_of(p, e, r);
    }
  }
}

// Exclusive scan of src[0..E) (shared memory) into dst[0..E], dst[E] = the
// total, by one warp; dst may be src.  Lane l takes a contiguous run.
__device__ __forceinline__ void warp_exclusive_scan(const int* src, int E, int* dst) {
  const int lane = threadIdx.x & 31;
  const int per = (E + 31) / 32;
  const int lo = min(lane * per, E), hi = min(lo + per, E);
  int sum = 0;
  for (int e = lo; e < hi; ++e) sum += src[e];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - sum;
  for (int e = lo; e < hi; ++e) {
    const int c = src[e];
    dst[e] = run;
    run += c;
  }
  if (lane == 31) dst[E] = incl;
  __syncwarp();
}

// The E-sized outputs, by one warp of CTA 0.  The counts (and f, P) are read
// in batches of eight loads per lane in flight, and the counts kept in the
// shared-memory scratch s_cnt[0..E) for the offsets and the rank loads.
template <int MODE>
__device__ __forceinline__ void finalize_warp(const RouterParams& p, const int32_t* counts, int* s_cnt) {
  const int lane = threadIdx.x & 31;
  const int E = p.E, k = p.k;
  constexpr bool kFwd = (MODE & kModeFwd) != 0, kDisp = (MODE & kModeDispatch) != 0;
  constexpr bool kHasP = kFwd && (MODE & kModeSplit) == 0;   // a split step writes P and the balance at its end
  // Sums of f*P, of squared count deviations and the extremes.  A deviation
  // c*E - T*k is exact in 64-bit integers; its square and the sums are fp32
  // (positive terms, relative error well under 1e-6 at E <= 1024).
  const long long tk = p.T * k;
  float fp = 0.f, dev = 0.f;
  int cmax = 0, cmin = 0x7fffffff, dropped = 0;
  constexpr int kB = 8;
  for (int e0 = 0; e0 < E; e0 += kB * kWarp) {
    int c[kB];
    float fv[kB], pv[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int e = e0 + j * kWarp + lane;
      c[j] = e < E ? __ldcg(counts + e) : 0;
      fv[j] = kHasP && e < E ? __ldcg(p.f + e) : 0.f;
      pv[j] = kHasP && e < E ? __ldcg(p.P + e) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int e = e0 + j * kWarp + lane;
      if (e < E) {
        s_cnt[e] = c[j];
        if constexpr (kDisp) {
          const int lower = p.cap_base != nullptr ? __ldg(p.cap_base + e) : 0;
          const int kept = min(c[j], max(p.C - lower, 0));
          p.kept[e] = kept;
          dropped += c[j] - kept;
        }
        if constexpr (kFwd) {
          fp = fmaf(fv[j], pv[j], fp);
          const float d = float((long long)c[j] * E - tk);
          dev = fmaf(d, d, dev);
          cmax = max(cmax, c[j]);
          cmin = min(cmin, c[j]);
        }
      }
    }
  }
  __syncwarp();
  if constexpr (kDisp) {
    warp_exclusive_scan(s_cnt, E, p.offsets);
    dropped = __reduce_add_sync(0xffffffffu, dropped);
    if (lane == 0) *p.n_dropped = dropped;
  }
  if constexpr (kFwd) {
    fp = warp_sum_f(fp);
    dev = warp_sum_f(dev);
    cmax = __reduce_max_sync(0xffffffffu, cmax);
    cmin = __reduce_min_sync(0xffffffffu, cmin);
    const int R = p.n_ranks;
    float rdev = 0.f;
    int rmax = 0;
    if (R > 0) {
      const int per = E / R;
      for (int r = lane; r < R; r += kWarp) {
        int load = 0;
        for (int j = 0; j < per; ++j) load += s_cnt[r * per + j];
        p.rank_load[r] = load;
        const float d = float((long long)load * R - tk);
        rdev = fmaf(d, d, rdev);
        rmax = max(rmax, load);
      }
      rdev = warp_sum_f(rdev);
      rmax = __reduce_max_sync(0xffffffffu, rmax);
    }
    if (lane == 0) {
      // mean = T*k/E; std/mean = sqrt(sum d^2 / E) / E / mean = sqrt(sum d^2) / (sqrt(E) * T*k)
      const float ftk = float(tk);
      if constexpr (kHasP) {
        const float balance = float(E) * fp;
        p.scalars[0] = p.alpha * balance;
        p.scalars[1] = balance;
      }
      p.scalars[2] = __fdiv_rn(__fsqrt_rn(dev), __fsqrt_rn(float(E)) * ftk);
      p.scalars[3] = __fdiv_rn(float(cmax) * float(E), ftk);
      p.scalars[4] = __fdiv_rn(float(cmin) * float(E), ftk);
      if (R > 0) {
        p.scalars[5] = __fdiv_rn(__fsqrt_rn(rdev), __fsqrt_rn(float(R)) * ftk);
        p.scalars[6] = __fdiv_rn(float(rmax) * float(R), ftk);
      } else {
        p.scalars[5] = 0.f;
        p.scalars[6] = 0.f;
      }
    }
  }
  // The extended step's bias update ([P1] §4.3): b_e + gamma * sign(T*k/E -
  // count_e), the sign taken exactly as sign(T*k - count_e * E), in fp32.
  // Every CTA read the bias before the grid barrier, so bias_out may alias it.
  if constexpr ((MODE & kModeExt) != 0) {
    if (p.bias_out != nullptr) {
      for (int e = lane; e < E; e += kWarp) {
        const long long d = tk - (long long)s_cnt[e] * E;
        const float dir = d > 0 ? 1.f : (d < 0 ? -1.f : 0.f);
        p.bias_out[e] = (p.bias != nullptr ? p.bias[e] : 0.f) + p.bias_gamma * dir;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// One warp of the CTA that counted itself done last: every other CTA has
// written its per-expert outputs and read the group sums.  Clears the group
// sums and the count for the next launch and writes the E-sized outputs.
// ---------------------------------------------------------------------------
template <int MODE>
__device__ __forceinline__ void finalize_last(const RouterParams& p, const int32_t* counts, int* s_cnt) {
  const int lane = threadIdx.x & 31;
  const int n = p.n_groups * p.E;
  for (int i = lane; i < n; i += kWarp) p.group_hist[i] = 0;
  if (lane == 0) p.ctrl->done = 0ull;
  finalize_warp<MODE>(p, counts, s_cnt);
}

// ---------------------------------------------------------------------------
// The dispatch warp after the forward: once the grid barrier has passed
// (bounded wait) it adds up the per-CTA sums of p of this CTA's experts (e =
// cta mod G) and counts the CTA done once the CTA's totals and bases are in
// shared memory; in the CTA that counts itself done last it then writes the
// E-sized outputs (shared-memory scratch s_cnt).  In the fused step it turns
// the in-CTA ranks into final positions, in chunks that the consumers done with
// the backward share.
// ---------------------------------------------------------------------------
// Waits (bounded) until this CTA's phase word reaches at_least or turns -1
// (an error elsewhere in the CTA); returns it, or -1 after recording an
// expired wait.  The limit is four times the wait limit: whatever the phase
// word waits for (the grid barrier, the CTA's own syncs) is bounded by the
// wait limit itself and reports its own expiry first.
__device__ __forceinline__ int wait_phase(const RouterParams& p, const int* s_phase, int at_least) {
  int ph = 0;
  uint64_t t0 = 0;
  for (unsigned spin = 0; (ph = *reinterpret_cast<const volatile int*>(s_phase)) >= 0 && ph < at_least; ++spin) {
    if ((spin & 15u) == 15u) {
      const uint64_t now = global_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > 4 * p.timeout_ns) {
        if ((threadIdx.x & 31) == 0) ctrl_set_error(p.ctrl, kErrPipelineTimeout);
        return -1;
      }
    }
    __nanosleep(64);
  }
  return ph;
}

// Final dispatch positions of the CTA's picks [a0, a0 + n) in chunks of
// kFixupChunk taken from the shared counter *s_next, by one warp; every warp
// that calls it takes chunks until none are left.
__device__ __forceinline__ void fixup_chunks(const RouterParams& p, long long a0, int n, const uint16_t* s_aidx,
                                             const uint16_t* s_arank, const int* s_off, const int* s_base, int* s_next) {
  const int lane = threadIdx.x & 31;
  const int n_chunks = (n + kFixupChunk - 1) / kFixupChunk;
  for (;;) {
    int c = 0;
    if (lane == 0) c = atomicAdd(s_next, 1);
    c = __shfl_sync(0xffffffffu, c, 0);
    if (c >= n_chunks) break;
    const int lo = c * kFixupChunk, len = min(kFixupChunk, n - lo);
    dispatch_fixup_smem(p, a0 + lo, len, s_aidx + lo, s_arank + lo, s_off, s_base);
  }
}

template <int MODE, bool STAGED>
__device__ __forceinline__ void dispatch_phase_c(const RouterParams& p, int cta, long long a0, long long a1, int* s_coff,
                                                 int* s_cbase, int* s_phase, const int32_t* counts, bool ranked,
                                                 const uint16_t* s_aidx, const uint16_t* s_arank, int* s_cnt,
                                                 int* s_next) {
  const int lane = threadIdx.x & 31;
  const int E = p.E;
  if (wait_phase(p, s_phase, 1) < 1) return;            // an error (or a lost signal): write nothing
  if constexpr ((MODE & kModeFwd) != 0 && (MODE & kModeSplit) == 0) {
    for (int e = cta; e < E; e += p.G) {
      const float Ps = warp_column_sum_f(p.P_part + (size_t)e * p.G_stride, p.G);
      if (lane == 0) p.P[e] = __fdiv_rn(Ps, (MODE & kModeExt) != 0 && p.masked_p ? float(p.T * p.k) : float(p.T));
    }
  }
  if (wait_phase(p, s_phase, 2) < 2) return;
  // counted done (release: this CTA's outputs; acquire: everyone else's, for the last)
  unsigned long long before = 0;
  if (lane == 0) before = atom_add_acq_rel_u64(&p.ctrl->done, 1ull);
  const bool last = __shfl_sync(0xffffffffu, before, 0) == (unsigned long long)(p.G - 1);
  __syncwarp();
  if constexpr ((MODE & kModeDispatch) != 0 && (MODE & kModeFwd) != 0) {   // given idx: the consumer warps do it
    warp_exclusive_scan(s_coff, E, s_coff);             // totals -> offsets
    if (lane == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile int*>(s_phase) = ranked ? 3 : 4;   // 3: the consumers may help with the chunks
    }
    __syncwarp();
    if (last) finalize_last<MODE>(p, counts, s_cnt);
    if (ranked) {
      if (s_aidx != nullptr) fixup_chunks(p, a0, int(a1 - a0), s_aidx, s_arank, s_coff, s_cbase, s_next);
      else if constexpr (STAGED) dispatch_fixup(p, p.idx, a0, a1, s_coff, s_cbase);
      else dispatch_direct(p, p.idx, a0, a1, s_coff, s_cbase);
    }
  } else {
    if (last) finalize_last<MODE>(p, counts, s_cnt);
  }
  trace_point(p, kTrDispatchDone);
}

// ---------------------------------------------------------------------------
// Ring bookkeeping.  With n stages and NS slots, slot q holds the stages
// s = q (mod NS); count_a(q) of them pass through it in the forward, whose fill
// of stage s is the slot's full-barrier completion s / NS.  In the backward the
// stage rel >= 1 slot-rounds below the slot's last stage is its refill rel - 1:
// full-barrier completion count_a(q) + rel - 1, issued after the consumption
// of the previous occupant, empty-barrier completion count_a(q) + rel - 1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ring_count_a(int q, int n, int NS) { return q < n ? (n - 1 - q) / NS + 1 : 0; }
__device__ __forceinline__ int ring_last(int q, int n, int NS) { return q + (ring_count_a(q, n, NS) - 1) * NS; }

// ---------------------------------------------------------------------------
// The persistent kernel.  MODE selects the phases:
//   A: per-CTA counts (and, with kModeFwd, idx/gate and sums of p), published
//      per CTA and into the group sums; then the launch's one grid barrier
//   C: per-expert totals, this CTA's dispatch bases and f (one round of L2
//      reads), P of the CTA's own experts, dispatch scatter (kModeDispatch),
//      backward (kModeBwd), and the E-sized outputs (scalars, rank loads,
//      offsets, kept, drops) written by the CTA that finishes its part last.
// STAGED: logit rows are 16-byte multiples and the producer warp streams them
// through the ring; otherwise the consumers read global memory directly.
// Launched cooperatively with p.G CTAs of kThreads threads.
// ---------------------------------------------------------------------------
template <class DT, int LPR, int VW, int NV, int NR, int MODE, bool STAGED, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) router_persistent_kernel(const RouterParams p) {
  using Raw = typename DT::Raw;
  constexpr int EPL = VW * NV;
  constexpr int RPW = kWarp / LPR;
  extern __shared__ __align__(128) unsigned char smem[];
  const int E = p.E, k = p.k, G = p.G, cta = blockIdx.x, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane / LPR, l = lane % LPR;
  const int S = STAGED ? p.rows_per_stage : 1;
  const int NS = STAGED ? p.n_slots : 1;
  const int stage_elems = S * E;
  constexpr bool kExt = (MODE & kModeExt) != 0;
  using PKey = typename PickKeyOf<kExt, typename DT::Key>::type;
  const SmemLayout L = router_smem_layout(E, int(sizeof(PKey)), STAGED ? NS : 0, stage_elems * int(sizeof(Raw)),
                                          p.asg_cap, p.rstat_cap);
  int* s_red = reinterpret_cast<int*>(smem + L.red);
  int* s_prog = s_red + kRedProg;     // stages finished per consumer warp (forward)
  int* s_phase = s_red + kRedPhase;
  int* s_ranked = s_red + kRedRanked;
  int* s_hist = reinterpret_cast<int*>(smem + L.hist);
  int* s_off = reinterpret_cast<int*>(smem + L.off);
  int* s_rank = reinterpret_cast<int*>(smem + L.rank);
  float* s_wf = reinterpret_cast<float*>(smem + L.w);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kMaxSlots;
  Raw* ring = reinterpret_cast<Raw*>(smem + L.ring);
  PKey* s_pick_w = reinterpret_cast<PKey*>(smem + L.pick) + warp * kPickSlotsPerWarp;

  const long long r0 = p.T * cta / G, r1 = p.T * (cta + 1) / G;
  const long long a0 = r0 * k, a1 = r1 * k;
  const int n_rows = int(r1 - r0);
  const int n_st = STAGED ? (n_rows + S - 1) / S : 0;
  const Raw* X = static_cast<const Raw*>(p.logits);
  int32_t* counts_dst = (MODE & kModeFwd) ? p.counts : p.counts_ws;
  // the CTA's dispatch in shared memory when its assignments fit
  // (also for a dispatch of given assignments, which loads them there)
  const bool asg_smem = ((STAGED && (MODE & kModeFwd) != 0) || MODE == kModeDispatch) && (MODE & kModeDispatch) != 0 &&
                        a1 - a0 <= p.asg_cap;
  uint16_t* s_aidx = asg_smem ? reinterpret_cast<uint16_t*>(smem + L.asg) : nullptr;
  uint16_t* s_arank = asg_smem ? s_aidx + p.asg_cap : nullptr;
  // each row's softmax statistics from the forward, for the backward
  float2* s_rstat = STAGED && (MODE & kModeFwd) != 0 && (MODE & kModeBwd) != 0 && r1 - r0 <= p.rstat_cap
                        ? reinterpret_cast<float2*>(smem + L.rstat) : nullptr;
  const bool is_producer = STAGED && warp == kProducerWarp && lane == 0;
  int fills[kMaxSlots];          // copies issued per slot (producer thread), drained on an error exit
  bool ranked = true;            // dispatch warp: every in-CTA rank of this CTA has been written
  // small CTAs: the consumers write the final dispatch positions, before the backward
  // the fused step's final dispatch positions: shared by the dispatch warp and
  // the consumers that are done with the backward, when the picks are in
  // shared memory
  const bool share_fixup = s_aidx != nullptr && (MODE & kModeFwd) != 0 && (MODE & kModeBwd) != 0;
#pragma unroll
  for (int q = 0; q < kMaxSlots; ++q) fills[q] = 0;

  for (int e = tid; e < E; e += kThreads) {
    s_hist[e] = 0;
    s_rank[e] = 0;
  }
  // per-consumer-warp expert counts (dispatch of given idx), or sums of the
  // picks' p (extended step with masked P)
  if constexpr ((MODE & kModeFwd) == 0 || kExt)
    for (int i = tid; i < kConsumerWarps * E; i += kThreads) reinterpret_cast<int*>(s_wf)[i] = 0;
  if (tid < kConsumerWarps) s_prog[tid] = 0;
  if (tid == 0) {
    *s_phase = 0;
    *s_ranked = 0;
    s_red[kRedFixNext] = 0;
    s_red[kRedCandReady] = 0;
    s_red[kRedCandDone] = 0;
  }
  if (STAGED && tid == 0) {
    for (int q = 0; q < NS; ++q) {
      mbar_init(&full[q], 1);
      mbar_init(&empty[q], kConsumerWarps);
    }
    mbar_fence_init();
  }
  // Launched with programmatic dependent launch, this grid may start while the
  // previous kernel of the stream is finishing: nothing above touches global
  // memory, and this waits until that kernel has completed and its writes are
  // visible (it returns at once otherwise).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  trace_point(p, kTrStart);
  __syncthreads();

  // ---- phase A
  if constexpr ((MODE & kModeFwd) != 0) {
    if (warp < kConsumerWarps) {
      float pacc[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) pacc[i] = 0.f;
      // the selection bias of the lane's columns (extended step; zero past E)
      float bl[EPL];
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VW; ++i) {
          const int c = col_of<LPR, VW>(v, l, i);
          bl[v * VW + i] = kExt && p.bias != nullptr && c < E ? __ldg(p.bias + c) : 0.f;
        }
      float* s_pm = s_wf + warp * E;                 // masked P: this warp's sums of the picks' p
      if constexpr (STAGED) {
        // The fast top-k path (bf16 rows of 32 lanes, at most 16 elements per lane).
        constexpr bool kFast = kFastTopk<DT, LPR, VW, NV> && !kExt;
        FastTopk<(EPL / 2 > 0 ? EPL / 2 : 1)> fs;
        fs.state = kFast && n_st > 1 ? 0 : 2;
        fs.tries = 0;
        fs.fails = 0;
        for (int s = 0; s < n_st; ++s) {
          const int q = s % NS;
          if (!mbar_wait(&full[q], (s / NS) & 1, p.timeout_ns)) {
            ctrl_set_error(p.ctrl, kErrPipelineTimeout);
            break;
          }
          if (s == 0) trace_point(p, kTrFirstStage);
          const Raw* st = ring + q * stage_elems;
          const int rows_here = min(S, n_rows - s * S);
          if constexpr (kFast) {
            if (fs.state == 1 && fs.tries >= 64) {
              if (fs.fails * 8 > fs.tries) fs.state = 2;      // more than one row in eight fails: stop trying
              fs.tries = 0;
              fs.fails = 0;
            }
            // The first stage's column sums choose the candidate set: each warp
            // adds its slice of the columns (into warp 0's slot of the per-warp
            // partials, unused until warp 0's rows are done) and the last warp
            // to finish chooses, while the others go on with their rows.
            if (s == 0 && n_st > 1) {
              stage_column_sums(reinterpret_cast<const uint16_t*>(st), rows_here, E, warp, reinterpret_cast<float*>(s_wf));
              __syncwarp();
              int last = 0;
              if (lane == 0) {
                __threadfence_block();
                last = atomicAdd(&s_red[kRedCandDone], 1) == kConsumerWarps - 1;
              }
              if (__shfl_sync(0xffffffffu, last, 0)) {
                __threadfence_block();
                choose_candidates(reinterpret_cast<const float*>(s_wf), E, s_red);
              }
            }
            fwd_stage_fast<DT, VW, NV, NR, (MODE & kModeSplit) == 0>(p, st, rows_here, r0 + (long long)s * S, warp, l,
                                                                     s_hist, pacc, s_pick_w, s_aidx, a0, s_rstat, r0, fs,
                                                                     s_red);
          } else {
            for (int sg = warp; sg * NR * RPW < rows_here; sg += kConsumerWarps) {
              const Raw* rows[NR];
              long long ts[NR];
              bool valids[NR];
#pragma unroll
              for (int r = 0; r < NR; ++r) {
                const int ri = (sg * NR + r) * RPW + g;
                valids[r] = ri < rows_here;
                rows[r] = st + (valids[r] ? ri : 0) * E;
                ts[r] = r0 + (long long)s * S + ri;
              }
              if constexpr (kExt)
                fwd_groups_ext<DT, LPR, VW, NV, NR, false>(p, rows, ts, valids, l, s_hist, pacc, s_pick_w, s_aidx, a0,
                                                           s_rstat, r0, bl, s_pm);
              else
                fwd_groups<DT, LPR, VW, NV, NR, false>(p, rows, ts, valids, l, s_hist, pacc, s_pick_w, s_aidx, a0,
                                                       s_rstat, r0);
            }
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&empty[q]);
            if constexpr ((MODE & kModeDispatch) != 0) {
              __threadfence_block();                        // idx stores before the progress mark
              *reinterpret_cast<volatile int*>(&s_prog[warp]) = s + 1;
            }
          }

        }
      } else {
        for (long long base = r0 + (long long)warp * NR * RPW; base < r1; base += (long long)kConsumerWarps * NR * RPW) {
          const Raw* rows[NR];
          long long ts[NR];
          bool valids[NR];
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            ts[r] = base + r * RPW + g;
            valids[r] = ts[r] < r1;
            rows[r] = X + (valids[r] ? ts[r] : r0) * (long long)E;
          }
          if constexpr (kExt)
            fwd_groups_ext<DT, LPR, VW, NV, NR, true>(p, rows, ts, valids, l, s_hist, pacc, s_pick_w, nullptr, 0,
                                                      nullptr, 0, bl, s_pm);
          else
            fwd_groups<DT, LPR, VW, NV, NR, true>(p, rows, ts, valids, l, s_hist, pacc, s_pick_w, nullptr, 0, nullptr, 0);
        }
      }
      trace_point(p, kTrFwdRows);
      trace_last(p, kTrFwdRowsAll);
      // Sum the row groups of the warp; group 0 stores the warp's partials
      // (a split step forms p in the backward instead).
#pragma unroll
      for (int i = 0; i < EPL; ++i)
#pragma unroll
        for (int off = LPR; off < kWarp; off <<= 1) pacc[i] += __shfl_xor_sync(0xffffffffu, pacc[i], off);
      if ((MODE & kModeSplit) == 0 && !(kExt && p.masked_p) && g == 0) {
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int i = 0; i < VW; ++i) {
            const int c = col_of<LPR, VW>(v, l, i);
            if (c < E) s_wf[warp * E + c] = pacc[v * VW + i];
          }
      }
    } else if (is_producer) {
      const uint64_t pol = l2_policy_evict_last();
      const uint32_t row_bytes = uint32_t(E) * uint32_t(sizeof(Raw));
      for (int s = 0; s < n_st; ++s) {
        const int q = s % NS;
        if (s >= NS && !mbar_wait(&empty[q], ((s / NS) - 1) & 1, p.timeout_ns)) {
          ctrl_set_error(p.ctrl, kErrPipelineTimeout);
          break;
        }
        const int rows_here = min(S, n_rows - s * S);
        const uint32_t bytes = uint32_t(rows_here) * row_bytes;
        mbar_arrive_expect_tx(&full[q], bytes);
        bulk_g2s(ring + q * stage_elems, X + (r0 + (long long)s * S) * E, bytes, &full[q], pol);
        ++fills[q];
      }
    } else if (STAGED && (MODE & kModeDispatch) != 0 && warp == kDispatchWarp) {
      // in-CTA dispatch ranks, one stage behind the consumer warps
      ranked = false;
      for (int s = 0; s < n_st; ++s) {
        bool ready = false;
        uint64_t t0 = 0;
        for (unsigned spin = 0; !ready; ++spin) {
          const int pr = lane < kConsumerWarps ? *reinterpret_cast<volatile int*>(&s_prog[lane]) : s + 1;
          ready = __all_sync(0xffffffffu, pr > s);
          if (!ready) {
            __nanosleep(256);                     // leave the issue slots to the consumer warps
            if ((spin & 15u) == 15u) {
              const uint64_t now = global_ns();
              if (t0 == 0) t0 = now;
              else if (now - t0 > p.timeout_ns) break;
            }
          }
        }
        if (!ready) {
          if (lane == 0) ctrl_set_error(p.ctrl, kErrPipelineTimeout);
          break;
        }
        __threadfence_block();
        const long long lo = (r0 + (long long)s * S) * k;
        const long long hi = min(r0 + (long long)(s + 1) * S, r1) * k;
        if (s_aidx != nullptr) local_ranks_smem(s_aidx, int(lo - a0), int(hi - a0), s_rank, s_arank);
        else local_ranks<kLoadOwn>(p.idx, lo, hi, E, s_rank, p.slot);
        if (s == n_st - 1) ranked = true;
      }
      if (n_st == 0) ranked = true;
      if (lane == 0) {
        __threadfence_block();                       // the ranks before the flag
        *reinterpret_cast<volatile int*>(s_ranked) = ranked ? 1 : -1;
      }
      trace_point(p, kTrRanked);
    }
  } else {
    // Dispatch of given assignments: consumer warp w ranks the w-th contiguous
    // chunk of this CTA's assignments (ranks within the chunk into s_arank, or
    // slot[] when the CTA's assignments do not fit in shared memory; counts per
    // expert in its row of s_wcnt); a prefix over the warps then gives each
    // chunk's base per expert and the CTA's counts.
    if (s_aidx != nullptr && warp != kDispatchWarp) {   // the CTA's expert ids, once, into shared memory
      constexpr int kB = 8;                          // loads per thread in flight together
      for (long long b0 = a0 + tid; b0 < a1; b0 += (long long)kB * kMainThreads) {
        int v[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const long long a = b0 + (long long)j * kMainThreads;
          v[j] = a < a1 ? __ldg(p.idx_in + a) : 0;
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const long long a = b0 + (long long)j * kMainThreads;
          if (a < a1) s_aidx[a - a0] = uint16_t(min(max(v[j], 0), E - 1));
        }
      }
      sync_main();                                   // the main group (the dispatch warp is not in it)
    }
    trace_point(p, kTrFirstStage);                   // the assignments are loaded
    if (warp < kConsumerWarps) {
      const long long n = a1 - a0;
      const long long lo = a0 + n * warp / kConsumerWarps, hi = a0 + n * (warp + 1) / kConsumerWarps;
      int* wcnt = reinterpret_cast<int*>(s_wf) + warp * E;
      if (s_aidx != nullptr) local_ranks_smem(s_aidx, int(lo - a0), int(hi - a0), wcnt, s_arank);
      else local_ranks<kLoadInput>(p.idx_in, lo, hi, E, wcnt, p.slot);
      trace_point(p, kTrFwdRows);
      trace_last(p, kTrFwdRowsAll);
    }
  }
  // Phase C shared memory: per expert f, the total (then the offsets) and this
  // CTA's base.  With the forward they take the per-warp partials' space, which
  // is spent after the publication below; a dispatch of given assignments
  // keeps its per-warp counts there and uses the offset and rank arrays.
  float* s_f = s_wf;
  int* s_coff = (MODE & kModeFwd) != 0 ? reinterpret_cast<int*>(s_wf + E) : s_off;
  int* s_cbase = (MODE & kModeFwd) != 0 ? s_coff + E + 1 : s_rank;
  if (warp == kDispatchWarp) {
    dispatch_phase_c<MODE, STAGED>(p, cta, a0, a1, s_coff, s_cbase, s_phase, counts_dst, ranked, s_aidx, s_arank,
                                   s_hist, s_red + kRedFixNext);
    return;
  }
  sync_main();
  if constexpr ((MODE & kModeFwd) == 0) {
    int* s_wcnt = reinterpret_cast<int*>(s_wf);
    for (int e = tid; e < E; e += kMainThreads) {
      int tot = 0;
#pragma unroll 1
      for (int w = 0; w < kConsumerWarps; ++w) {
        const int c = s_wcnt[w * E + e];
        s_wcnt[w * E + e] = tot;
        tot += c;
      }
      s_hist[e] = tot;
    }
    sync_main();
  }
  // Publish this CTA's counts (per CTA, and into its group's sums) and sums of p.
  {
    int32_t* grp_hist = p.group_hist + (size_t)(cta / kGroupCtas) * E;
    for (int e = tid; e < E; e += kMainThreads) {
      const int c = s_hist[e];
      p.tile_hist[(size_t)e * p.G_stride + cta] = c;
      if (c != 0) atomicAdd(grp_hist + e, c);
      if constexpr ((MODE & kModeFwd) != 0 && (MODE & kModeSplit) == 0) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) t += s_wf[w * E + e];
        p.P_part[(size_t)e * p.G_stride + cta] = t;
      }
    }
  }
  trace_point(p, kTrFwdDone);
  if (!grid_barrier(p.ctrl, G, p.barrier_extra, 1, true, p.timeout_ns, s_red + kRedFlag, kBarMain, kMainThreads)) {
    if (tid == 0) *reinterpret_cast<volatile int*>(s_phase) = -1;
    if (is_producer)   // let every issued copy land before the CTA exits
      for (int q = 0; q < NS; ++q)
        if (fills[q] > 0) mbar_wait(&full[q], (fills[q] - 1) & 1, kDrainNs);
    return;
  }
  if (tid == 0) {
    __threadfence_block();
    *reinterpret_cast<volatile int*>(s_phase) = 1;      // the dispatch warp may add up its experts' p
    // The next kernel of the stream may be scheduled as SMs free up; it waits
    // for this grid's completion before it touches memory.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  trace_point(p, kTrBarrier1);

  // ---- phase C
  // Per expert: the total over all CTAs, f, and this CTA's base; the CTA that
  // owns expert e (e = cta mod G) writes its count and f.
  totals_and_bases(p, cta, s_coff, s_cbase);
  sync_main();
  for (int e = tid; e < E; e += kMainThreads) {
    const int total = s_coff[e];
    const float fe = __fdiv_rn(float(total), float(p.T * k));
    if constexpr ((MODE & kModeFwd) != 0) s_f[e] = fe;
    if (e % G == cta) {             // ordered before the dispatch warp's done count by the syncs below
      counts_dst[e] = total;
      if constexpr ((MODE & kModeFwd) != 0) p.f[e] = fe;
    }
  }
  sync_main();
  if (warp == 0) {
    // the offsets: here for a dispatch of given assignments, else by the dispatch warp
    if constexpr ((MODE & kModeFwd) == 0) warp_exclusive_scan(s_coff, E, s_coff);
    if (lane == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile int*>(s_phase) = 2;    // totals (offsets) and bases are in shared memory
    }
  }
  sync_main();
  trace_point(p, kTrScanDone);
  if constexpr ((MODE & kModeFwd) == 0) {
    // final positions of the given assignments, chunk by chunk
    if (warp < kConsumerWarps) {
      const int* s_wcnt = reinterpret_cast<const int*>(s_wf) + warp * E;
      const long long n = a1 - a0;
      const long long lo = a0 + n * warp / kConsumerWarps, hi = a0 + n * (warp + 1) / kConsumerWarps;
      constexpr int kB = 8;                                // assignments per lane in flight together
      for (long long b0 = lo; b0 < hi; b0 += kB * kWarp) {
        int e_[kB], loc_[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const long long a = b0 + j * kWarp + lane;
          if (s_aidx != nullptr) {
            e_[j] = a < hi ? int(s_aidx[a - a0]) : 0;
            loc_[j] = a < hi ? int(s_arank[a - a0]) : 0;
          } else {
            e_[j] = a < hi ? min(max(__ldg(p.idx_in + a), 0), E - 1) : 0;
            loc_[j] = a < hi ? __ldcg(p.slot + a) : 0;
          }
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const long long a = b0 + j * kWarp + lane;
          const int e = e_[j];
          const int r = s_cbase[e] + s_wcnt[e] + loc_[j];
          if (a < hi && r >= 0 && r < s_coff[e + 1] - s_coff[e]) {   // always true for consistent ranks
            p.perm[s_coff[e] + r] = int(a);
            p.slot[a] = slot_of(p, e, r);
          }
        }
      }
    }
  }
  if constexpr ((MODE & kModeBwd) != 0) {
    const float coef = p.grad_scale * p.alpha * float(E) / float(p.T);
    // extended step: the dense aux coefficient (zero with masked P, whose aux
    // term reaches the picks only) and the picks' one, g*alpha*E/(T*k)
    const float coef_f = kExt && p.masked_p ? 0.f : coef;
    const float coef_m = p.grad_scale * p.alpha * float(E) / float(p.T * k);
    if (warp < kConsumerWarps) {
      float fr[EPL];
      load_f<LPR, VW, NV>(s_f, E, l, coef_f, fr);
      constexpr bool kSplit = (MODE & kModeSplit) != 0;
      static_assert(!kSplit || (STAGED && kFastTopk<DT, LPR, VW, NV>), "split steps run on the fast variants");
      float pacc_b[EPL];                           // a split step's sums of p over the warp's rows
#pragma unroll
      for (int i = 0; i < EPL; ++i) pacc_b[i] = 0.f;
      if constexpr (STAGED) {
        for (int s = n_st - 1; s >= 0; --s) {
          const int q = s % NS;
          const int rel = (ring_last(q, n_st, NS) - s) / NS;     // 0: still in the ring from the forward
          if (rel > 0 && !mbar_wait(&full[q], (ring_count_a(q, n_st, NS) + rel - 1) & 1, p.timeout_ns)) {
            ctrl_set_error(p.ctrl, kErrPipelineTimeout);
            break;
          }
          if (s == n_st - 1) trace_point(p, kTrBwdFirst);
          const Raw* st = ring + q * stage_elems;
          const int rows_here = min(S, n_rows - s * S);
          // extended step: with one row per warp (32 lanes per row) the gate
          // terms of the warp's rows of the stage are formed ahead into its pick
          // slots when they fit (E = 384: 296 -> 286 us per step); else, and
          // with several rows per warp, whose per-row work is shared anyway,
          // each row group's upstream gate gradients are loaded one group ahead
          const float* gp_pre = nullptr;
          float dg_next = 0.f;
          if constexpr (kExt) {
            const int per = kConsumerWarps * RPW;
            const int n_rows_w = rows_here > warp * RPW ? (rows_here - warp * RPW + per - 1) / per * RPW : 0;
            if (LPR == kWarp && s_rstat != nullptr && n_rows_w * kMaxK <= kPickSlotsPerWarp) {
              float* gp_buf = reinterpret_cast<float*>(s_pick_w);
              __syncwarp();
              ext_gate_prepass<DT, LPR>(p, st, r0 + (long long)s * S, s * S, rows_here, warp, n_rows_w, s_rstat,
                                        s_aidx, a0, coef_m, s_f, gp_buf);
              gp_pre = gp_buf;
            } else {
              dg_next = dgate_of(p, r0 + (long long)s * S + warp * RPW + g, l, warp * RPW + g < rows_here);
            }
          }
          for (int gi = warp; gi * RPW < rows_here; gi += kConsumerWarps) {
            const int ri = gi * RPW + g;
            const bool valid = ri < rows_here;
            float dg_cur = 0.f;
            if constexpr (kExt) {
              if (gp_pre == nullptr) {
                dg_cur = dg_next;
                const int rn = (gi + kConsumerWarps) * RPW + g;
                dg_next = dgate_of(p, r0 + (long long)s * S + rn, l, rn < rows_here);
              }
            }
            Raw raw[EPL];
            load_lane<DT, LPR, VW, NV, false>(st + (valid ? ri : 0) * E, E, l, valid, raw);
            if constexpr (kSplit) {
              float mx;
              if (s_rstat != nullptr) {
                mx = s_rstat[valid ? s * S + ri : 0].x;
              } else {
                float m = -3.402823466e38f;
#pragma unroll
                for (int i = 0; i < EPL; ++i) m = fmaxf(m, __uint_as_float(DT::bits(raw[i])));
                mx = group_max<LPR>(m);
              }
              bwd_group_split<DT, LPR, VW, NV>(raw, fr, r0 + (long long)s * S + ri, valid, l, E, mx, pacc_b, p.dlogits);
              if constexpr (kSplitGatesInBwd<EPL>)
                split_gates<DT, LPR>(p, st + (valid ? ri : 0) * E, r0 + (long long)s * S + ri, valid, l, mx, s_aidx, a0);
            } else {
              float mx, inv_s;
              if (s_rstat != nullptr) {
                const float2 rs = s_rstat[valid ? s * S + ri : 0];
                mx = rs.x;
                inv_s = rs.y;
              } else {
                bwd_row_stats<DT, LPR, VW, NV>(raw, mx, inv_s);
              }
              if constexpr (kExt)
                bwd_group_ext<DT, LPR, VW, NV, false>(p, raw, st + (valid ? ri : 0) * E, fr, r0 + (long long)s * S + ri,
                                                      valid, l, E, mx, inv_s, coef_f, coef_m, s_f, s_aidx, a0, dg_cur,
                                                      gp_pre, (gi - warp) / kConsumerWarps * RPW + g);
              else
                bwd_group<DT, LPR, VW, NV>(raw, fr, r0 + (long long)s * S + ri, valid, l, E, mx, inv_s, p.dlogits);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[q]);
        }
      } else {
        const long long n_groups = (r1 - r0 + RPW - 1) / RPW;
        for (long long gi = n_groups - 1 - warp; gi >= 0; gi -= kConsumerWarps) {
          const long long t = r0 + gi * RPW + g;
          const bool valid = t < r1;
          Raw raw[EPL];
          load_lane<DT, LPR, VW, NV, true>(X + (valid ? t : r0) * (long long)E, E, l, valid, raw);
          float mx, inv_s;
          bwd_row_stats<DT, LPR, VW, NV>(raw, mx, inv_s);
          if constexpr (kExt)
            bwd_group_ext<DT, LPR, VW, NV, true>(p, raw, X + (valid ? t : r0) * (long long)E, fr, t, valid, l, E, mx,
                                                 inv_s, coef_f, coef_m, s_f, nullptr, 0, dgate_of(p, t, l, valid),
                                                 nullptr, 0);
          else
            bwd_group<DT, LPR, VW, NV>(raw, fr, t, valid, l, E, mx, inv_s, p.dlogits);
        }
      }
      trace_point(p, kTrBwdRows);
      trace_last(p, kTrBwdRowsAll);
      if constexpr (kSplit) {
        // This CTA's sums of p: each warp's into the ring's memory (free once
        // every consumer is past the backward), added over the warps in a
        // fixed order, then into the fixed-point totals.  The CTA that adds
        // its sums last writes P, the balance and L_aux, and clears the totals.
        float* s_pw = reinterpret_cast<float*>(ring);      // [kConsumerWarps][E]
        named_barrier(kBarConsumers, kConsumerThreads);
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int i = 0; i < VW; ++i) {
            const int c = col_of<LPR, VW>(v, l, i);
            if (c < E) s_pw[warp * E + c] = pacc_b[v * VW + i];
          }
        named_barrier(kBarConsumers, kConsumerThreads);
        for (int c = tid; c < E; c += kConsumerThreads) {
          float t = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) t += s_pw[w * E + c];
          pfix_add(p.pfix + c, p.pfix + kMaxExperts + c, t);
        }
        __threadfence();
        named_barrier(kBarConsumers, kConsumerThreads);
        if (tid == 0) s_red[kRedBwdLast] = atom_add_acq_rel_u64(&p.ctrl->bwd_done, 1ull) == (unsigned long long)(G - 1);
        named_barrier(kBarConsumers, kConsumerThreads);
        if (s_red[kRedBwdLast]) {
          __threadfence();
          for (int c = tid; c < E; c += kConsumerThreads) {
            const double tot = pfix_value(__ldcg(p.pfix + c), __ldcg(p.pfix + kMaxExperts + c));
            const float Pc = float(tot / double(p.T));
            p.P[c] = Pc;
            s_pw[c] = Pc;
            p.pfix[c] = 0ull;
            p.pfix[kMaxExperts + c] = 0ull;
          }
          named_barrier(kBarConsumers, kConsumerThreads);
          if (warp == 0) {
            float fp = 0.f;
            for (int c = lane; c < E; c += kWarp) fp = fmaf(__ldcg(p.f + c), s_pw[c], fp);
            fp = warp_sum_f(fp);
            if (lane == 0) {
              const float balance = float(E) * fp;
              p.scalars[0] = p.alpha * balance;
              p.scalars[1] = balance;
              p.ctrl->bwd_done = 0ull;
            }
          }
        }
      }
      // then help with the final dispatch positions that remain
      if (share_fixup && wait_phase(p, s_phase, 3) == 3)
        fixup_chunks(p, a0, int(a1 - a0), s_aidx, s_arank, s_coff, s_cbase, s_red + kRedFixNext);
    } else if (is_producer) {
      const uint64_t pol = l2_policy_evict_first();
      const uint32_t row_bytes = uint32_t(E) * uint32_t(sizeof(Raw));
      for (int s = n_st - NS - 1; s >= 0; --s) {
        const int q = s % NS;
        const int rel = (ring_last(q, n_st, NS) - s) / NS;       // >= 1 here
        if (!mbar_wait(&empty[q], (ring_count_a(q, n_st, NS) + rel - 1) & 1, p.timeout_ns)) {
          ctrl_set_error(p.ctrl, kErrPipelineTimeout);
          break;
        }
        const int rows_here = min(S, n_rows - s * S);
        const uint32_t bytes = uint32_t(rows_here) * row_bytes;
        mbar_arrive_expect_tx(&full[q], bytes);
        bulk_g2s(ring + q * stage_elems, X + (r0 + (long long)s * S) * E, bytes, &full[q], pol);
        ++fills[q];
      }
    }
  }
  sync_main();
  trace_point(p, kTrJoined);
  // Every copy was waited on by the consumers in a normal run (these tests then
  // pass at once); after an expired wait this keeps the CTA until its copies land.
  if (is_producer)
    for (int q = 0; q < NS; ++q)
      if (fills[q] > 0) mbar_wait(&full[q], (fills[q] - 1) & 1, kDrainNs);
  trace_point(p, kTrEnd);
}

// Backward alone: a plain grid-stride streaming kernel (8 warps of 256-thread CTAs).
template <class DT, int LPR, int VW, int NV>
__global__ void __launch_bounds__(256) router_bwd_kernel(const BwdParams p) {
  using Raw = typename DT::Raw;
  constexpr int EPL = VW * NV;
  constexpr int RPW = kWarp / LPR;
  __shared__ float s_f[1024];
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) s_f[e] = __ldg(p.f + e);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int g = lane / LPR, l = lane % LPR;
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long nw = (long long)gridDim.x * 8;
  const Raw* X = static_cast<const Raw*>(p.logits);
  float fr[EPL];
  load_f<LPR, VW, NV>(s_f, p.E, l, p.coef, fr);
  for (long long base = gw * RPW; base < p.T; base += nw * RPW) {
    const long long t = base + g;
    const bool valid = t < p.T;
    Raw raw[EPL];
    load_lane<DT, LPR, VW, NV, true>(X + (valid ? t : 0) * (long long)p.E, p.E, l, valid, raw);
    float mx, inv_s;
    bwd_row_stats<DT, LPR, VW, NV>(raw, mx, inv_s);
    bwd_group<DT, LPR, VW, NV>(raw, fr, t, valid, l, p.E, mx, inv_s, p.dlogits);
  }
}

}  // namespace moe
