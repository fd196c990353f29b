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
// The kernel is bound by HBM bandwidth.  The columns of a head's state are
// independent given the token's keys and query (every reduction runs over the
// key index d), so a CTA owns one head and one slab of 32 value columns: a
// 16 KB slice of the state, read once into registers (float4 per thread, 8
// threads per row, 16 row groups) and written once.  The key/query dot
// products are recomputed per slab (a few hundred flops).  Small CTAs let
// several slices per SM be in their load phase while others compute and
// store.  Loads and stores use the streaming cache hint: every byte of the
// state is touched once per call.
//
// With a channel-wise gate alpha (KDA, the family table of "08 · linear
// 路线（三）" §1.4: S <- (I - beta k k^T) Diag(alpha) S + beta k v^T), the
// decayed state Diag(alpha) S0 takes the place of g S0: r_j = S0^T (alpha *
// k_j), r_q = S0^T (alpha * q), S' = Diag(alpha) S0 + sum_j beta_j k_j e_j^T.
//
// With the input prologue on (delta_step_prologue), the raw q and k of the
// token go through SiLU and an L2 norm over the key index and beta through
// sigmoid or 2 sigmoid ("DeltaProduct" §2.2; the query path of the layer
// design in "08 · linear 路线（三）" §3) in shared memory, before any of the
// above: no extra pass over HBM.
#include <cuda_bf16.h>

#include "kernels.h"

namespace delta {
namespace {

constexpr int kThreads = 128;
constexpr int kSlab = 32;      // value columns per CTA (fewer when dv < 32)
constexpr int kMaxD = 128;
constexpr int kMaxRows = 8;    // state rows per thread at dk = 128

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

__device__ __forceinline__ float silu(float x) { return x / (1.f + __expf(-x)); }

template <int NH, bool KDA>
__global__ void __launch_bounds__(kThreads, 6) step_kernel(StepArgs a) {
  __shared__ float s_k[NH][kMaxD];
  __shared__ float s_q[kMaxD];
  __shared__ float s_v[NH][kSlab];
  __shared__ float s_e[NH][kSlab];
  __shared__ float s_r[NH + 1][kSlab];
  __shared__ float s_beta[NH];
  __shared__ float s_dot[NH + 1][NH];  // [i][j] = k_i.k_j (i<j); [NH][j] = k_j.q
  __shared__ float s_inv[NH + 1];      // prologue: 1 / ||SiLU(k_j)||, 1 / ||SiLU(q)||
  __shared__ float s_alpha[kMaxD];     // channel-wise gate (KDA)
  // partial sums per row group: (NH + 1) x RG x SW floats, RG * SW == 4 * kThreads
  // (written as float4: 16-byte alignment)
  __shared__ __align__(16) float s_part[(NH + 1) * 4 * kThreads];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int dk = a.dk, dv = a.dv;
  const int SW = dv < kSlab ? dv : kSlab;
  const int nslab = dv / SW;
  const int64_t bh = blockIdx.x / nslab;
  const int cbase = (blockIdx.x % nslab) * SW;
  const int64_t b = bh / a.H, h = bh % a.H, H = a.H;

  // ---- the state slice: thread owns 4 columns of rows d = rg, rg + RG, ... ----
  const int tpr = SW / 4;          // threads per row
  const int RG = kThreads / tpr;   // row groups
  const int rg = tid / tpr;
  const int c4 = (tid % tpr) * 4;  // column within the slab
  float4 *srow = reinterpret_cast<float4 *>(a.state + bh * (int64_t)dk * dv + cbase);
  float4 S[kMaxRows];
#pragma unroll
  for (int i = 0; i < kMaxRows; ++i) {
    const int d = rg + i * RG;
    if (d < dk) S[i] = __ldcs(srow + ((int64_t)d * dv + c4) / 4);
  }

  // ---- token inputs to shared memory ----
  for (int i = tid; i < dk; i += kThreads) s_q[i] = load_io(a.q, bh * dk + i, a.bf16);
  for (int i = tid; i < NH * dk; i += kThreads) {
    const int j = i / dk, d = i % dk;
    s_k[j][d] = load_io(a.k, ((b * NH + j) * H + h) * dk + d, a.bf16);
  }
  for (int i = tid; i < NH * SW; i += kThreads) {
    const int j = i / SW, c = i % SW;
    s_v[j][c] = load_io(a.v, ((b * NH + j) * H + h) * dv + cbase + c, a.bf16);
  }
  if (tid < NH) {
    const float x = a.beta[(b * NH + tid) * H + h];
    s_beta[tid] = a.beta_map < 0 ? x : (a.beta_map == 1 ? 2.f : 1.f) / (1.f + __expf(-x));
  }
  constexpr bool kda = KDA;  // channel-wise gate a.alpha (else the scalar a.g)
  if (kda)
    for (int i = tid; i < dk; i += kThreads) s_alpha[i] = a.alpha[bh * dk + i];
  const float gate = kda ? 1.0f : (a.g ? a.g[bh] : 1.0f);
  __syncthreads();  // token inputs visible
  if (a.beta_map >= 0) {
    // ---- prologue: q, k_j <- SiLU(.) / ||SiLU(.)||_2 (0 for a zero vector) ----
    for (int i = tid; i < (NH + 1) * dk; i += kThreads) {
      float *p = i < NH * dk ? &s_k[i / dk][i % dk] : &s_q[i - NH * dk];
      *p = silu(*p);
    }
    __syncthreads();
    for (int j = warp; j <= NH; j += kThreads / 32) {
      const float *p = j < NH ? s_k[j] : s_q;
      float ss = 0.f;
      for (int d = lane; d < dk; d += 32) ss = fmaf(p[d], p[d], ss);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_inv[j] = ss > 0.f ? rsqrtf(ss) : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < (NH + 1) * dk; i += kThreads) {
      if (i < NH * dk)
        s_k[i / dk][i % dk] *= s_inv[i / dk];
      else
        s_q[i - NH * dk] *= s_inv[NH];
    }
    __syncthreads();
  }

  // ---- the small dot products k_i.k_j and k_j.q, one warp each ----
  {
    int pair = 0;
#pragma unroll
    for (int j = 0; j < NH; ++j) {
#pragma unroll
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
            s_dot[NH][j] = acc;
        }
      }
    }
  }

  // ---- partial r_j = S0^T k_j and r_q = S0^T q over this thread's rows ----
  float4 part[NH + 1];
#pragma unroll
  for (int j = 0; j <= NH; ++j) part[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kMaxRows; ++i) {
    const int d = rg + i * RG;
    if (d < dk) {
      const float ad = kda ? s_alpha[d] : 1.0f;  // the row's decay (KDA)
#pragma unroll
      for (int j = 0; j <= NH; ++j) {
        const float w = ((j < NH) ? s_k[j][d] : s_q[d]) * ad;
        part[j].x = fmaf(S[i].x, w, part[j].x);
        part[j].y = fmaf(S[i].y, w, part[j].y);
        part[j].z = fmaf(S[i].z, w, part[j].z);
        part[j].w = fmaf(S[i].w, w, part[j].w);
      }
    }
  }
  // s_part layout: [j][rg][SW]
#pragma unroll
  for (int j = 0; j <= NH; ++j)
    *reinterpret_cast<float4 *>(s_part + ((size_t)j * RG + rg) * SW + c4) = part[j];
  __syncthreads();
  for (int i = tid; i < (NH + 1) * SW; i += kThreads) {
    const int j = i / SW, c = i % SW;
    const float *src = s_part + (size_t)j * RG * SW + c;
    float acc = 0.0f;
    const int rows_used = dk < RG ? dk : RG;
    for (int r = 0; r < rows_used; ++r) acc += src[(size_t)r * SW];
    s_r[j][c] = acc;
  }
  __syncthreads();

  // ---- prediction errors and the output, per value column ----
  for (int c = tid; c < SW; c += kThreads) {
    float o = gate * s_r[NH][c];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      float pred = gate * s_r[j][c];
#pragma unroll
      for (int i = 0; i < j; ++i) pred = fmaf(s_beta[i] * s_dot[i][j], s_e[i][c], pred);
      const float e = s_v[j][c] - pred;
      s_e[j][c] = e;
      o = fmaf(s_beta[j] * s_dot[NH][j], e, o);
    }
    store_io(a.out, bh * dv + cbase + c, o, a.bf16);
  }
  __syncthreads();

  // ---- S' = g S0 + sum_j beta_j k_j e_j^T, written in place ----
  float4 be[NH];
#pragma unroll
  for (int j = 0; j < NH; ++j)
    be[j] = make_float4(s_beta[j] * s_e[j][c4], s_beta[j] * s_e[j][c4 + 1],
                        s_beta[j] * s_e[j][c4 + 2], s_beta[j] * s_e[j][c4 + 3]);
#pragma unroll
  for (int i = 0; i < kMaxRows; ++i) {
    const int d = rg + i * RG;
    if (d < dk) {
      const float gd = kda ? s_alpha[d] : gate;
      float4 x = make_float4(S[i].x * gd, S[i].y * gd, S[i].z * gd, S[i].w * gd);
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const float kd = s_k[j][d];
        x.x = fmaf(kd, be[j].x, x.x);
        x.y = fmaf(kd, be[j].y, x.y);
        x.z = fmaf(kd, be[j].z, x.z);
        x.w = fmaf(kd, be[j].w, x.w);
      }
      __stcs(srow + ((int64_t)d * dv + c4) / 4, x);
    }
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs &a, cudaStream_t s) {
  const int sw = a.dv < kSlab ? a.dv : kSlab;
  const unsigned grid = (unsigned)(a.B * a.H * (a.dv / sw));
  const bool kda = a.alpha != nullptr;
  switch (a.n_h) {
    case 1: (kda ? step_kernel<1, true> : step_kernel<1, false>)<<<grid, kThreads, 0, s>>>(a); break;
    case 2: (kda ? step_kernel<2, true> : step_kernel<2, false>)<<<grid, kThreads, 0, s>>>(a); break;
    case 3: (kda ? step_kernel<3, true> : step_kernel<3, false>)<<<grid, kThreads, 0, s>>>(a); break;
    case 4: (kda ? step_kernel<4, true> : step_kernel<4, false>)<<<grid, kThreads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace delta
