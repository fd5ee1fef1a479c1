// Device helpers shared by the router kernels: order-preserving top-k keys,
// lane-group reductions, the bounded grid barrier and exp2.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kWarp = 32;
constexpr float kLog2e = 1.4426950408889634f;   // log2(e)

// ---------------------------------------------------------------------------
// Workspace control block (first 256 bytes of the caller's workspace).
// ---------------------------------------------------------------------------
struct Ctrl {
  unsigned bar_count;   // CTAs arrived at the current grid barrier (0 between barriers)
  unsigned bar_gen;     // barrier generation, bumped by the last arriver
  int error;            // sticky error bits, read and cleared by the host
  int pad[61];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");

enum : int { kErrBarrierTimeout = 1 };

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_volatile_i32(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

// Grid-wide barrier for a cooperative launch (all CTAs co-resident).  The wait
// is bounded by `timeout_ns`; on expiry the CTA records kErrBarrierTimeout.
// Returns false (uniformly across the CTA) once any CTA of the launch has
// recorded an error: the caller must then stop writing and return, and later
// barriers stop waiting because the flag is already set.
__device__ __forceinline__ bool grid_barrier(Ctrl* c, unsigned nblocks, uint64_t timeout_ns, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned gen = ld_acquire_u32(&c->bar_gen);
    __threadfence();
    const unsigned arrived = atomicAdd(&c->bar_count, 1u);
    if (arrived == nblocks - 1) {
      atomicExch(&c->bar_count, 0u);
      __threadfence();
      atomicAdd(&c->bar_gen, 1u);
    } else {
      const uint64_t t0 = global_ns();
      while (ld_acquire_u32(&c->bar_gen) == gen) {
        if (ld_volatile_i32(&c->error) != 0) break;
        if (global_ns() - t0 > timeout_ns) {
          atomicOr(&c->error, kErrBarrierTimeout);
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
    *s_flag = ld_volatile_i32(&c->error);
  }
  __syncthreads();
  return *s_flag == 0;
}

// ---------------------------------------------------------------------------
// exp2 on the special-function unit (flush-to-zero): the hardware instruction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Element types.  Raw is the storage word of one element.
// ---------------------------------------------------------------------------
struct Bf16 {
  using Raw = uint16_t;
  using Key = int;          // 32-bit: 16 value bits + 16 index bits
  static __device__ __forceinline__ float to_float(Raw r) { return __uint_as_float(uint32_t(r) << 16); }
  // Order-preserving signed key: larger logit -> larger key; equal logits ->
  // the lower column has the larger key.  -0.0 and +0.0 map to the same value.
  static __device__ __forceinline__ Key key(Raw r, int col) {
    const int s = int(uint32_t(r) << 16);
    const int v = s < 0 ? -(s & 0x7fffffff) : s;   // sign-magnitude -> two's complement
    return v | (0xffff - col);                        // low 16 bits of v are zero
  }
  static __device__ __forceinline__ int key_col(Key k) { return 0xffff - (k & 0xffff); }
  static __device__ __forceinline__ float key_value(Key k) {
    const int v = k & int(0xffff0000u);
    const uint32_t bits = v < 0 ? (0x80000000u | uint32_t(-v)) : uint32_t(v);
    return __uint_as_float(bits);
  }
  static constexpr Key kKeyMin = int(0x80000000u);
};

struct Fp32 {
  using Raw = uint32_t;
  using Key = long long;    // 64-bit: 32 value bits + 32 index bits
  static __device__ __forceinline__ float to_float(Raw r) { return __uint_as_float(r); }
  static __device__ __forceinline__ Key key(Raw r, int col) {
    const int s = int(r);
    const long long v = s < 0 ? -(long long)(s & 0x7fffffff) : (long long)s;
    return (long long)((unsigned long long)v << 32) | (long long)(0xffffffffu - uint32_t(col));
  }
  static __device__ __forceinline__ int key_col(Key k) { return int(0xffffffffu - uint32_t(k & 0xffffffffll)); }
  static __device__ __forceinline__ float key_value(Key k) {
    const long long v = k >> 32;    // arithmetic shift: the signed magnitude
    const uint32_t bits = v < 0 ? (0x80000000u | uint32_t(-v)) : uint32_t(v);
    return __uint_as_float(bits);
  }
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
__device__ __forceinline__ int group_max_key(int x) {
  if constexpr (LPR == 32) {
    return __reduce_max_sync(0xffffffffu, x);
  } else {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
  }
}

template <int LPR>
__device__ __forceinline__ long long group_max_key(long long x) {
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) {
    const long long y = __shfl_xor_sync(0xffffffffu, x, off);
    x = y > x ? y : x;
  }
  return x;
}

// Deterministic block-wide sum (fixed order) of one float per thread.
template <int NT>
__device__ __forceinline__ float block_sum(float x, float* scratch /* >= NT/32 floats */) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  __syncthreads();
  if (lane == 0) scratch[w] = x;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t += scratch[i];
  return t;
}

}  // namespace moe
