// tc_common.cuh -- small device helpers shared by the two tensor-core
// kernels of the chunked forward (the UT-transform pass and the state pass).
#pragma once

#include <cstdint>

#include "sm100.cuh"

namespace delta {
namespace tc {

constexpr float kLog2e = 1.4426950408889634f;
// log g is clamped here, so that g = 0 (a reset) stays finite
constexpr float kLogGateFloor = -80.0f;
// Down to this cumulative log2 gate within a chunk the decay factors are
// formed as 2^gc_i * 2^-gc_j (no overflow); below it, exactly per entry.
constexpr float kRatioFloor = -100.0f;

// 2^x on the MUFU unit (relative error ~2^-22; flushes to 0 far below 1)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2 g of a gate g in [0, 1], clamped at kLogGateFloor nats: lg2 on the
// MUFU unit (absolute error ~2^-22 near 1; g = 0 and subnormal g give the
// floor).  A short body: the gate scan runs in every chunk of the state pass.
__device__ __forceinline__ float gate_log2(float g) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(g));
  return fmaxf(y, kLogGateFloor * kLog2e);
}

// Named barrier over 128 threads.
__device__ __forceinline__ void named_sync(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// Named barrier over 128 threads that also ORs `cond` across them, so that
// every participant takes the same decision (used to leave a loop together
// once any role has aborted).
__device__ __forceinline__ bool named_sync_or(int id, bool cond) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %2, 0;\n\t"
      "bar.red.or.pred q, %1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"((uint32_t)cond)
      : "memory");
  return r != 0;
}

// One arrival per warp once every lane's prior work (fenced by the caller) is
// done: the warp converges, then lane 0 arrives.
__device__ __forceinline__ void arrive_warp(uint64_t *bar, int lane) {
  __syncwarp();
  if (lane == 0) sm100::mbar_arrive(bar);
}

// Inclusive prefix sum over the 64 log-gate entries of a chunk, per warp:
// lane holds entries lane and lane + 32.
__device__ __forceinline__ void warp_scan64(const float *lam, int lane, float &lo, float &hi) {
  lo = lam[lane];
  hi = lam[lane + 32];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float a = __shfl_up_sync(0xffffffffu, lo, o);
    const float c = __shfl_up_sync(0xffffffffu, hi, o);
    if (lane >= o) {
      lo += a;
      hi += c;
    }
  }
  hi += __shfl_sync(0xffffffffu, lo, 31);
}

}  // namespace tc
}  // namespace delta
