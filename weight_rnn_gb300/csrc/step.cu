// step.cu -- one decode token of Gated DeltaProduct (n_h >= 1 sub-steps) for
// every (b, h), with the float32 state resident in HBM and updated in place.
//
// The recurrence of "DeltaProduct：通过 Householder 乘积增强线性 RNN 的状态追踪"
// §2.6 for one token -- S <- g S, then for j: e_j = v_j - S^T k_j,
// S <- S + beta_j k_j e_j^T, then o = S^T q -- is rearranged so that the state
// is read exactly once and written exactly once.  With S0 the incoming state
// and r_j = S0^T k_j, r_q = S0^T q (all reductions over the key index done in
// the single read pass):
//
//   e_1 = v_1 - g r_1
//   e_j = v_j - (g r_j + sum_{i<j} beta_i (k_i . k_j) e_i)
//   o   = g r_q + sum_j beta_j (k_j . q) e_j
//   S'  = g S0 + sum_j beta_j k_j e_j^T
//
// (expand S after each sub-step: S_j = g S0 + sum_{i<=j} beta_i k_i e_i^T, so
// S_{j-1}^T k_j and S_{n_h}^T q are the sums above).
//
// The kernel is bound by HBM bandwidth: one CTA per (b, h) head, each row of
// the state is read by float4 loads across a warp (dv/4 threads per row) and
// held in registers between the read and the write; the reductions over the
// key index use shared memory across row groups.  Loads and stores of the
// state use the streaming cache hint: every byte is touched once per call.
#include <cuda_bf16.h>

#include "kernels.h"

namespace delta {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxNh = 4;
constexpr int kMaxD = 128;
constexpr int kMaxRows = 16;  // rows of the state held per thread (dk = 128, dv = 128)

__device__ __forceinline__ float load_io(const void *p, int64_t i, bool bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i])
              : static_cast<const float *>(p)[i];
}

__device__ __forceinline__ void store_io(void *p, int64_t i, float x, bool bf16) {
  if (bf16)
    static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
  else
    static_cast<float *>(p)[i] = x;
}

__global__ void __launch_bounds__(kThreads, 2) step_kernel(StepArgs a) {
  __shared__ float s_k[kMaxNh][kMaxD];
  __shared__ float s_q[kMaxD];
  __shared__ float s_v[kMaxNh][kMaxD];
  __shared__ float s_e[kMaxNh][kMaxD];
  __shared__ float s_r[kMaxNh + 1][kMaxD];
  __shared__ float s_beta[kMaxNh];
  __shared__ float s_dot[kMaxNh + 1][kMaxNh];  // [i][j] = k_i.k_j (i<j); [n_h][j] = k_j.q
  // partial sums per row group: (n_h + 1) x RG x dv floats, RG * dv == 4 * kThreads
  __shared__ float s_part[(kMaxNh + 1) * 4 * kThreads];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dk = a.dk, dv = a.dv, n_h = a.n_h;
  const int64_t bh = blockIdx.x;
  const int64_t b = bh / a.H, h = bh % a.H, H = a.H;

  // ---- token inputs to shared memory ----
  for (int i = tid; i < dk; i += kThreads) s_q[i] = load_io(a.q, bh * dk + i, a.bf16);
  for (int i = tid; i < n_h * dk; i += kThreads) {
    const int j = i / dk, d = i % dk;
    s_k[j][d] = load_io(a.k, ((b * n_h + j) * H + h) * dk + d, a.bf16);
  }
  for (int i = tid; i < n_h * dv; i += kThreads) {
    const int j = i / dv, c = i % dv;
    s_v[j][c] = load_io(a.v, ((b * n_h + j) * H + h) * dv + c, a.bf16);
  }
  if (tid < n_h) s_beta[tid] = a.beta[(b * n_h + tid) * H + h];
  const float gate = a.g ? a.g[bh] : 1.0f;

  // ---- the state: thread owns 4 columns of rows d = rg, rg + RG, ... ----
  const int tpr = dv / 4;          // threads per row
  const int RG = kThreads / tpr;   // row groups
  const int rg = tid / tpr;
  const int c4 = (tid % tpr) * 4;
  float4 *srow = reinterpret_cast<float4 *>(a.state + bh * (int64_t)dk * dv);
  float4 S[kMaxRows];
#pragma unroll
  for (int i = 0; i < kMaxRows; ++i) {
    const int d = rg + i * RG;
    if (d < dk) S[i] = __ldcs(srow + ((int64_t)d * dv + c4) / 4);
  }
  __syncthreads();  // token inputs visible

  // ---- the small dot products k_i.k_j and k_j.q, one warp each ----
  {
    int pair = 0;
    for (int j = 0; j < n_h; ++j) {
      for (int i = 0; i <= j; ++i, ++pair) {
        // i < j: k_i.k_j ; i == j: k_j.q
        if (pair % (kThreads / 32) != warp) continue;
        float acc = 0.0f;
        for (int d = lane; d < dk; d += 32) acc += s_k[j][d] * (i < j ? s_k[i][d] : s_q[d]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
          if (i < j)
            s_dot[i][j] = acc;
          else
            s_dot[n_h][j] = acc;
        }
      }
    }
  }

  // ---- partial r_j = S0^T k_j and r_q = S0^T q over this thread's rows ----
  float4 part[kMaxNh + 1];
#pragma unroll
  for (int j = 0; j <= kMaxNh; ++j) part[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kMaxRows; ++i) {
    const int d = rg + i * RG;
    if (d < dk) {
#pragma unroll
      for (int j = 0; j <= kMaxNh; ++j) {
        if (j > n_h) continue;
        const float w = (j < n_h) ? s_k[j][d] : s_q[d];
        part[j].x = fmaf(S[i].x, w, part[j].x);
        part[j].y = fmaf(S[i].y, w, part[j].y);
        part[j].z = fmaf(S[i].z, w, part[j].z);
        part[j].w = fmaf(S[i].w, w, part[j].w);
      }
    }
  }
  // s_part layout: [j][rg][dv]
#pragma unroll
  for (int j = 0; j <= kMaxNh; ++j) {
    if (j > n_h) continue;
    float *dst = s_part + ((size_t)j * RG + rg) * dv + c4;
    dst[0] = part[j].x;
    dst[1] = part[j].y;
    dst[2] = part[j].z;
    dst[3] = part[j].w;
  }
  __syncthreads();
  for (int i = tid; i < (n_h + 1) * dv; i += kThreads) {
    const int j = i / dv, c = i % dv;
    const float *src = s_part + (size_t)j * RG * dv + c;
    float acc = 0.0f;
    const int rows_used = dk < RG ? dk : RG;
    for (int r = 0; r < rows_used; ++r) acc += src[(size_t)r * dv];
    s_r[j][c] = acc;
  }
  __syncthreads();

  // ---- prediction errors and the output, per value column ----
  for (int c = tid; c < dv; c += kThreads) {
    float o = gate * s_r[n_h][c];
    for (int j = 0; j < n_h; ++j) {
      float pred = gate * s_r[j][c];
      for (int i = 0; i < j; ++i) pred = fmaf(s_beta[i] * s_dot[i][j], s_e[i][c], pred);
      const float e = s_v[j][c] - pred;
      s_e[j][c] = e;
      o = fmaf(s_beta[j] * s_dot[n_h][j], e, o);
    }
    store_io(a.out, bh * dv + c, o, a.bf16);
  }
  __syncthreads();

  // ---- S' = g S0 + sum_j beta_j k_j e_j^T, written in place ----
  float4 be[kMaxNh];
#pragma unroll
  for (int j = 0; j < kMaxNh; ++j) {
    if (j < n_h)
      be[j] = make_float4(s_beta[j] * s_e[j][c4], s_beta[j] * s_e[j][c4 + 1],
                          s_beta[j] * s_e[j][c4 + 2], s_beta[j] * s_e[j][c4 + 3]);
  }
#pragma unroll
  for (int i = 0; i < kMaxRows; ++i) {
    const int d = rg + i * RG;
    if (d < dk) {
      float4 x = make_float4(S[i].x * gate, S[i].y * gate, S[i].z * gate, S[i].w * gate);
#pragma unroll
      for (int j = 0; j < kMaxNh; ++j) {
        if (j < n_h) {
          const float kd = s_k[j][d];
          x.x = fmaf(kd, be[j].x, x.x);
          x.y = fmaf(kd, be[j].y, x.y);
          x.z = fmaf(kd, be[j].z, x.z);
          x.w = fmaf(kd, be[j].w, x.w);
        }
      }
      __stcs(srow + ((int64_t)d * dv + c4) / 4, x);
    }
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs &a, cudaStream_t s) {
  step_kernel<<<(unsigned)(a.B * a.H), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace delta
