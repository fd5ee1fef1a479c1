// Device helpers shared by the router kernels: the bounded grid barrier,
// mbarrier / bulk-copy (TMA) primitives, order-preserving top-k keys, exp2
// and lane-group reductions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kWarp = 32;
constexpr float kLog2e = 1.4426950408889634f;   // log2(e)

// ---------------------------------------------------------------------------
// Workspace control block (first 512 bytes of the caller's workspace).
//
// The per-expert counts of each group of kGroupCtas consecutive CTAs are
// accumulated with integer atomics in the workspace right after this block
// (zero before a launch; CTA 0 clears them again at the end of the launch).
//
// One 64-bit word carries the grid-barrier arrival count (low half) and the
// sticky error bits (high half), so that an arrival is a single atomic and a
// waiter learns both "everyone is here" and "someone failed" from one load.
// The count grows by one per CTA and barrier during a launch; the last CTA to
// arrive at the launch's final barrier takes it back to 0.  A failed launch
// leaves the count wherever it stopped and the error bits set; the host reads
// and clears both (moe_get_device_status), and until then every later launch
// sees the error at its first barrier and writes nothing after it.
// ---------------------------------------------------------------------------
struct Ctrl {
  unsigned long long sync;      // [31:0] arrivals, [63:32] error bits
  unsigned long long done;      // CTAs whose per-expert outputs are written (the launch's CTA 0 resets it)
  unsigned long long bwd_done;  // CTAs of a split fused step that have added their sums of p (the last resets it)
  unsigned long long pad[61];
};
static_assert(sizeof(Ctrl) == 512, "control block is 512 bytes");

enum : int { kErrBarrierTimeout = 1, kErrPipelineTimeout = 2 };

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t) :: "memory");
  return t;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long atom_add_acq_rel_u64(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

__device__ __forceinline__ void ctrl_set_error(Ctrl* c, int bits) {
  atomicOr(&c->sync, (unsigned long long)(unsigned)bits << 32);
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Grid-wide barrier number `round` (1, 2, ...) of a cooperative launch (all
// CTAs co-resident).  It passes once the arrival count reaches
// round * (nblocks + extra); extra is 0 except in tests of the timeout path,
// where it makes the barrier unreachable.  On the launch's final barrier
// (`last`) the CTA that completes it subtracts the launch's arrivals again, and
// its waiters accept a count of 0 as passed.  Every wait is bounded by
// `timeout_ns`; on expiry the CTA records kErrBarrierTimeout.  Returns false
// (uniformly across the CTA) once any CTA of the launch, or of an earlier
// launch not yet cleared by the host, has recorded an error: the caller must
// then stop writing and return.
//
// Called by the `nthreads` threads (whole warps, including thread 0) that
// synchronise on named barrier `bar_id` within the CTA.
__device__ __forceinline__ bool grid_barrier(Ctrl* c, unsigned nblocks, unsigned extra, unsigned round, bool last,
                                             uint64_t timeout_ns, int* s_flag, int bar_id, int nthreads) {
  named_barrier(bar_id, nthreads);               // the group's writes happen before thread 0's arrival
  if (threadIdx.x == 0) {
    const unsigned target = (nblocks + extra) * round;
    const unsigned long long old = atom_add_acq_rel_u64(&c->sync, 1ull);
    unsigned err = unsigned(old >> 32);
    if (err == 0 && unsigned(old) + 1u == target) {
      if (last) atomicAdd(&c->sync, 0ull - (unsigned long long)target);   // back to 0 for the next launch
    } else if (err == 0) {
      uint64_t t0 = 0;
      for (unsigned spin = 0;; ++spin) {
        const unsigned long long v = ld_acquire_u64(&c->sync);
        err = unsigned(v >> 32);
        const unsigned n = unsigned(v);
        if (err != 0 || n >= target || (last && n == 0)) break;
        if ((spin & 15u) == 15u) {
          const uint64_t now = global_ns();
          if (t0 == 0) {
            t0 = now;
          } else if (now - t0 > timeout_ns) {
            ctrl_set_error(c, kErrBarrierTimeout);
            err = kErrBarrierTimeout;
            break;
          }
        }
        if (spin > 8) __nanosleep(32);
      }
    }
    *s_flag = int(err);
  }
  named_barrier(bar_id, nthreads);
  return *s_flag == 0;
}

// ---------------------------------------------------------------------------
// mbarrier and bulk asynchronous copy (TMA, non-tensor form).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Like mbar_test, but the thread may be suspended in hardware for up to
// `hint_ns` until the phase completes (no issue slots spent while waiting).
__device__ __forceinline__ bool mbar_test_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

// Waits until the barrier phase of parity `parity` has completed; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_test_suspend(bar, parity, 20000u)) {
    if (global_ns() - t0 > timeout_ns) return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to shared memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy) : "memory");
}

// ---------------------------------------------------------------------------
// exp2 on the special-function unit (flush-to-zero): the hardware instruction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes per instruction (Blackwell packed fp32): a*b, a+b, a*b+c,
// each rounded to nearest like the scalar operation.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "add.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%6, %7};\n\t"
      "fma.rn.f32x2 x, x, y, z;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Reciprocal on the special-function unit (the hardware instruction).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Element types.  Raw is the storage word of one element; bits() gives its
// fp32 bit pattern.  key_from_bits(b, lane_bits, elem_bits) is an
// order-preserving integer key of the value with bit pattern b in column
// lane_bits | elem_bits (two disjoint bit fields: the lane's share of the
// column and the element's): a larger logit gives a larger key, and of equal
// logits the lower column gets the larger key.
// ---------------------------------------------------------------------------
struct Bf16 {
  using Raw = uint16_t;
  // Unsigned: bit 31 set for values from +0 up, bits 16..30 the magnitude
  // (inverted for negative values), bits 0..15 the column inverted.  Built
  // with two instructions: a byte permute that replicates the sign into the
  // upper half and takes the lane's column bits into the lower half, then one
  // three-input logic op.  The one place where the key order differs from
  // the value order is -0.0, which ranks just below +0.0; callers that must
  // treat the two as equal check the picks with is_zero().
  using Key = uint32_t;
  static constexpr bool kSplitsZero = true;
  static constexpr Raw kNegInf = 0xff80u;
  static __device__ __forceinline__ uint32_t bits(Raw r) { return uint32_t(r) << 16; }
  static __device__ __forceinline__ Key key_from_bits(uint32_t b, uint32_t lane_bits, uint32_t elem_bits) {
    uint32_t s, k;
    asm("prmt.b32 %0, %1, %2, 0xBB54;" : "=r"(s) : "r"(b), "r"(lane_bits));
    // per bit: b ^ s where the constant is 0 (bits 16..30), s ^ c where b is 0
    // (bits 0..15), and NOT b at bit 31 (b and s both hold the sign there)
    asm("lop3.b32 %0, %1, %2, %3, 0x16;" : "=r"(k) : "r"(b), "r"(s), "r"(0x80000000u | (0xffffu ^ elem_bits)));
    return k;
  }
  static __device__ __forceinline__ int key_col(Key k) { return int(0xffffu ^ (k & 0xffffu)); }
  static __device__ __forceinline__ float key_value(Key k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fff0000u) : (~k & 0xffff0000u));
  }
  // +0.0 or -0.0
  static __device__ __forceinline__ bool is_zero(Key k) { return (k >> 16) - 0x7fffu <= 1u; }
  static __device__ __forceinline__ uint32_t canonical_zero(uint32_t b) { return b == 0x80000000u ? 0u : b; }
  static constexpr Key kKeyMin = 0u;
};

struct Fp32 {
  using Raw = uint32_t;
  using Key = long long;    // signed: 32 value bits (two's complement of the magnitude) above 32 column bits
  static constexpr bool kSplitsZero = false;
  static constexpr Raw kNegInf = 0xff800000u;
  static __device__ __forceinline__ uint32_t bits(Raw r) { return r; }
  static __device__ __forceinline__ Key key_from_bits(uint32_t b, uint32_t lane_bits, uint32_t elem_bits) {
    const uint32_t col = lane_bits | elem_bits;
    const int v = int(b);
    const int s = v >> 31;
    const long long m = (long long)((v ^ (s & 0x7fffffff)) - s);   // two's complement of the magnitude
    return (long long)((unsigned long long)m << 32) | (long long)(0xffffffffu - uint32_t(col));
  }
  static __device__ __forceinline__ int key_col(Key k) { return int(0xffffffffu - uint32_t(k & 0xffffffffll)); }
  static __device__ __forceinline__ float key_value(Key k) {
    const long long v = k >> 32;
    const uint32_t b = v < 0 ? (0x80000000u | uint32_t(-v)) : uint32_t(v);
    return __uint_as_float(b);
  }
  static __device__ __forceinline__ bool is_zero(Key) { return false; }
  static __device__ __forceinline__ uint32_t canonical_zero(uint32_t b) { return b; }
  static constexpr Key kKeyMin = (long long)0x8000000000000000ull;
};

// ---------------------------------------------------------------------------
// Reductions over a group of LPR consecutive lanes (LPR in {8, 16, 32}); every
// lane of the warp must call them.
// ---------------------------------------------------------------------------
template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

template <int LPR>
__device__ __forceinline__ float group_max(float x) {
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

template <int LPR>
__device__ __forceinline__ uint32_t group_max_key(uint32_t x) {
  if constexpr (LPR == 32) {
    return __reduce_max_sync(0xffffffffu, x);
  } else {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
  }
}

// 64-bit keys (Fp32: signed value word above the column word).  Over a whole
// warp: the largest value word, as an unsigned number with the sign bit
// flipped (the same order), by one warp reduction, then the largest column
// word among the lanes holding it by a second one.
template <int LPR>
__device__ __forceinline__ long long group_max_key(long long x) {
  if constexpr (LPR == 32) {
    const uint32_t hi = uint32_t((unsigned long long)x >> 32) ^ 0x80000000u;
    const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t lo = __reduce_max_sync(0xffffffffu, hi == mh ? uint32_t((unsigned long long)x) : 0u);
    return (long long)(((unsigned long long)(mh ^ 0x80000000u) << 32) | lo);
  } else {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) {
      const long long y = __shfl_xor_sync(0xffffffffu, x, off);
      x = y > x ? y : x;
    }
    return x;
  }
}

__device__ __forceinline__ float warp_sum_f(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

}  // namespace moe
