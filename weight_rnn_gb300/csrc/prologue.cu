// prologue.cu -- the input prologue of "DeltaProduct：通过 Householder 乘积增强
// 线性 RNN 的状态追踪" §2.2 (keys psi(.) / ||psi(.)||_2 with psi = SiLU, beta =
// phi(.) with phi = sigmoid or 2 sigmoid), with the query path of the layer
// design in "08 · linear 路线（三）：delta rule 与 DPLR 统一框架" §3 (SiLU then
// L2 norm, as for the keys).
//
// One pass, bound by HBM: every raw element is read once and its result
// written once.  A row of dk elements is spread over dk / V lanes that each
// load and store 16 bytes (V = 8 bf16 or 4 float32 values); the row's sum of
// squares is a shuffle reduction within that lane group.  The arithmetic is
// float32; a row whose SiLU is all zero stays zero.
#include <cuda_bf16.h>

#include "kernels.h"

namespace delta {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;  // rows in flight per lane group

// SiLU with two MUFU operations (exp and reciprocal, relative error ~2^-21):
// for float32 outputs
__device__ __forceinline__ float silu_f32(float x) { return __fdividef(x, 1.f + __expf(-x)); }
// SiLU with one, x sigmoid(x) = h + h tanh(h) with h = x / 2 (tanh.approx,
// relative error ~2^-11, below the bf16 rounding of the result): for bf16
// outputs, where the MUFU rate would otherwise bound the kernel
__device__ __forceinline__ float silu_bf16(float x) {
  const float h = 0.5f * x;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}
__device__ __forceinline__ float sigmoid(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

template <typename In>
__device__ __forceinline__ void unpack(const uint4 &u, float (&x)[16 / sizeof(In)]) {
  if constexpr (sizeof(In) == 2) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
  }
}

template <typename In>
__device__ __forceinline__ uint4 pack(const float (&x)[16 / sizeof(In)]) {
  if constexpr (sizeof(In) == 2) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
}

template <typename In>
__global__ void __launch_bounds__(kThreads) prologue_kernel(PrologueArgs a) {
  constexpr int V = 16 / sizeof(In);  // values per lane
  const int lpr = a.dk / V;            // lanes per row: a power of two in [2, 32]
  const int lane = threadIdx.x & 31;
  const int sub = lane % lpr;
  const int64_t rows = a.rows_q + a.rows_k;
  const int64_t rpw = 32 / lpr;  // rows per warp and load
  const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
  const int64_t gw = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  // kRows rows per lane group per round, their loads issued before any use
  // so that enough bytes are in flight to keep HBM busy
  for (int64_t base = gw * rpw * kRows; base < rows; base += warps * rpw * kRows) {
    uint4 u[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int64_t row = base + j * rpw + lane / lpr;
      const bool isq = row < a.rows_q;
      const int64_t r = isq ? row : row - a.rows_q;
      u[j] = make_uint4(0, 0, 0, 0);
      if (row < rows)
        u[j] = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const In *>(isq ? a.q : a.k) + r * a.dk) + sub);
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int64_t row = base + j * rpw + lane / lpr;
      const bool isq = row < a.rows_q;
      const int64_t r = isq ? row : row - a.rows_q;
      float x[V];
      unpack<In>(u[j], x);
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        x[i] = sizeof(In) == 2 ? silu_bf16(x[i]) : silu_f32(x[i]);
        ss = fmaf(x[i], x[i], ss);
      }
      // sum over the row's lane group (xor offsets below lpr stay inside it)
      for (int o = lpr >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) x[i] *= inv;
      if (row < rows)
        __stcs(reinterpret_cast<uint4 *>(static_cast<In *>(isq ? a.q_out : a.k_out) + r * a.dk) + sub,
               pack<In>(x));
    }
  }
  const float scale = a.beta_map == 1 ? 2.f : 1.f;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < a.n_beta;
       i += (int64_t)gridDim.x * kThreads)
    a.beta_out[i] = scale * sigmoid(__ldcs(a.beta + i));
}

}  // namespace

cudaError_t launch_prologue(const PrologueArgs &a, cudaStream_t s) {
  const int64_t rows = a.rows_q + a.rows_k;
  const int lpr = a.dk / (a.bf16 ? 8 : 4);
  const int64_t rows_per_block = (int64_t)(kThreads / 32) * (32 / lpr) * kRows;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // enough blocks to cover every row once, at most as many as are resident
  // at a time (grid-stride beyond that)
  auto kern = a.bf16 ? prologue_kernel<__nv_bfloat16> : prologue_kernel<float>;
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0)) != cudaSuccess)
    return e;
  int64_t grid = (rows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace delta
