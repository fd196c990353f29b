// diag.cu -- two diagnostics on the outputs of the forward pass, each one
// block per (b, h) on the CUDA cores in float32:
//
//   erank_kernel          the effective rank of a state matrix ("DeltaProduct：
//                         通过 Householder 乘积增强线性 RNN 的状态追踪" §4.6):
//                         erank(S) = exp(-sum_k p_k log p_k), p_k = sigma_k /
//                         sum_j sigma_j over the singular values of S
//   attention_map_kernel  the fully parallel form of "08 · linear 路线（三）：
//                         delta rule 与 DPLR 统一框架" §2.4 with the gated
//                         decay of §3, for one block of N <= 64 steps:
//                         A = (Q K^T * Gam * M) T with o_i = sum_j A_ij v_j
#include <cuda_bf16.h>

#include "kernels.h"

namespace delta {
namespace {

constexpr int kDiagThreads = 256;   // attention map
constexpr int kErankThreads = 1024; // effective rank: one warp per column pair, 2 pairs a step
constexpr int kMaxSweeps = 40;
// a column pair counts as orthogonal once |a.b| <= kOrthTol * |a| |b| (the error
// this leaves in the singular values is of the order of kOrthTol squared)
constexpr float kOrthTol = 1e-5f;
constexpr float kLogGateFloorNat = -80.0f;  // log g clamped here (g = 0 stays finite)

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// One-sided Jacobi SVD of S [dk][dv] (row-major in global memory): the dv
// columns, held column-major in shared memory, are rotated pairwise until
// every pair is orthogonal; the singular values are then the column norms.
// Pairs follow the round-robin (circle) schedule: in step s column 0 meets
// column L_{n-1}, and L_i meets L_{n-1-i}, with L_i = ((i - 1 + s) mod
// (n - 1)) + 1, so that each step rotates n/2 disjoint pairs (one warp per
// pair at a time) and n - 1 steps meet every pair once.
__global__ void __launch_bounds__(kErankThreads, 1)
erank_kernel(const float *__restrict__ S, float *__restrict__ erank, int dk, int dv) {
  extern __shared__ float cols[];  // [dv][dk]
  __shared__ int rotated;
  __shared__ float red[2][kErankThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nw = kErankThreads / 32;
  const float *Sm = S + (size_t)blockIdx.x * dk * dv;
  for (int idx = tid; idx < dk * dv; idx += kErankThreads) {
    const int r = idx / dv, c = idx % dv;
    cols[c * dk + r] = Sm[idx];
  }
  __syncthreads();
  const int n = dv, half = dv / 2;
  for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
    if (tid == 0) rotated = 0;
    __syncthreads();
    for (int s = 0; s < n - 1; ++s) {
      for (int i = warp; i < half; i += nw) {
        const int p = i == 0 ? 0 : ((i - 1 + s) % (n - 1)) + 1;
        const int q = ((n - 2 - i + s) % (n - 1)) + 1;
        float *a = cols + p * dk, *b = cols + q * dk;
        float al = 0.f, be = 0.f, ga = 0.f;
        for (int r = lane; r < dk; r += 32) {
          const float x = a[r], y = b[r];
          al = fmaf(x, x, al);
          be = fmaf(y, y, be);
          ga = fmaf(x, y, ga);
        }
        al = warp_sum(al);
        be = warp_sum(be);
        ga = warp_sum(ga);
        if (ga != 0.f && fabsf(ga) > kOrthTol * sqrtf(al) * sqrtf(be)) {
          // the rotation that zeroes a.b: tan of its angle is the smaller
          // root t of t^2 + 2 zeta t - 1 = 0, zeta = (b.b - a.a) / (2 a.b)
          const float zeta = (be - al) / (2.f * ga);
          const float t = copysignf(1.f, zeta) / (fabsf(zeta) + hypotf(1.f, zeta));
          const float c = rsqrtf(fmaf(t, t, 1.f)), sn = c * t;
          for (int r = lane; r < dk; r += 32) {
            const float x = a[r], y = b[r];
            a[r] = c * x - sn * y;
            b[r] = sn * x + c * y;
          }
          if (lane == 0) rotated = 1;
        }
      }
      __syncthreads();
    }
    const int any = rotated;
    __syncthreads();
    if (!any) break;
  }
  // sigma_c = |column c|; p_c = sigma_c / sum sigma; H = -sum p log p
  float sum = 0.f, plogp = 0.f;
  for (int c = warp; c < dv; c += nw) {
    float sq = 0.f;
    for (int r = lane; r < dk; r += 32) sq = fmaf(cols[c * dk + r], cols[c * dk + r], sq);
    sq = warp_sum(sq);
    const float sg = sqrtf(sq);
    sum += sg;
    plogp += sg > 0.f ? sg * logf(sg) : 0.f;  // sum sigma log sigma, normalised below
  }
  if (lane == 0) {
    red[0][warp] = sum;
    red[1][warp] = plogp;
  }
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f, sl = 0.f;
    for (int w = 0; w < nw; ++w) {
      tot += red[0][w];
      sl += red[1][w];
    }
    // -sum p log p with p = sigma / tot: log tot - (sum sigma log sigma) / tot
    erank[blockIdx.x] = tot > 0.f ? expf(logf(tot) - sl / tot) : 0.f;
  }
}

template <typename In>
__device__ __forceinline__ float ld(const In *p) {
  if constexpr (sizeof(In) == 2) return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
  else return *p;
}

// One block per (b, h): Q, K [N][dk] in shared memory as float32, the
// cumulative log gate gc, then
//   A_ij = beta_i (k_i . k_j) exp(gc_i - gc_j)   (i > j; masked before exp)
//   X    = (I + A)^{-1}  by column-oriented forward substitution (thread j
//          carries column j; at step k its entry k is final and the rows
//          below take -A_ik x_kj), T = X diag(beta)
//   P_il = (q_i . k_l) exp(gc_i - gc_l)  (l <= i)
//   attn_ij = sum_{j <= l <= i} P_il T_lj
template <typename In>
__global__ void __launch_bounds__(kDiagThreads)
attention_map_kernel(const In *__restrict__ q, const In *__restrict__ k,
                     const float *__restrict__ beta, const float *__restrict__ g,
                     float *__restrict__ attn, int H, int N, int dk) {
  extern __shared__ float sm[];
  float *Qs = sm;                 // [N][dk]
  float *Ks = Qs + N * dk;        // [N][dk]
  float *A = Ks + N * dk;         // [N][N]: A, then T
  float *X = A + N * N;           // [N][N]
  float *P = X + N * N;           // [N][N]
  float *gc = P + N * N;          // [N]
  float *bt = gc + N;             // [N]
  const int tid = threadIdx.x;
  const int bh = blockIdx.x, b = bh / H, h = bh % H;
  for (int idx = tid; idx < N * dk; idx += kDiagThreads) {
    const int t = idx / dk, d = idx % dk;
    const size_t off = (((size_t)b * N + t) * H + h) * dk + d;
    Qs[idx] = ld(q + off);
    Ks[idx] = ld(k + off);
  }
  for (int t = tid; t < N; t += kDiagThreads) bt[t] = beta[((size_t)b * N + t) * H + h];
  if (tid == 0) {
    float acc = 0.f;
    for (int t = 0; t < N; ++t) {
      if (g) acc += fmaxf(logf(g[((size_t)b * N + t) * H + h]), kLogGateFloorNat);
      gc[t] = acc;
    }
  }
  __syncthreads();
  // A (strictly lower) and P (lower incl. the diagonal); X = I
  for (int idx = tid; idx < N * N; idx += kDiagThreads) {
    const int i = idx / N, j = idx % N;
    float kk = 0.f, qk = 0.f;
    if (j <= i) {
      for (int d = 0; d < dk; ++d) {
        kk = fmaf(Ks[i * dk + d], Ks[j * dk + d], kk);
        qk = fmaf(Qs[i * dk + d], Ks[j * dk + d], qk);
      }
    }
    const float dec = j <= i ? expf(gc[i] - gc[j]) : 0.f;
    A[idx] = j < i ? bt[i] * kk * dec : 0.f;
    P[idx] = qk * dec;
    X[idx] = i == j ? 1.f : 0.f;
  }
  __syncthreads();
  if (tid < N) {
    const int j = tid;
    for (int kx = j; kx < N; ++kx) {
      const float xk = X[kx * N + j];
      for (int i = kx + 1; i < N; ++i) X[i * N + j] = fmaf(-A[i * N + kx], xk, X[i * N + j]);
    }
  }
  __syncthreads();
  for (int idx = tid; idx < N * N; idx += kDiagThreads) A[idx] = X[idx] * bt[idx % N];  // T
  __syncthreads();
  float *out = attn + (size_t)bh * N * N;
  for (int idx = tid; idx < N * N; idx += kDiagThreads) {
    const int i = idx / N, j = idx % N;
    float acc = 0.f;
    for (int l = j; l <= i; ++l) acc = fmaf(P[i * N + l], A[l * N + j], acc);
    out[idx] = acc;
  }
}

}  // namespace

int64_t erank_smem_bytes(int dk, int dv) { return (int64_t)dk * dv * 4; }

cudaError_t launch_erank(const float *state, float *erank, int64_t BH, int dk, int dv,
                         cudaStream_t s) {
  const int smem = (int)erank_smem_bytes(dk, dv);
  cudaError_t e = cudaFuncSetAttribute(erank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  erank_kernel<<<(unsigned)BH, kErankThreads, smem, s>>>(state, erank, dk, dv);
  return cudaGetLastError();
}

cudaError_t launch_attention_map(const void *q, const void *k, const float *beta, const float *g,
                                 float *attn, int64_t B, int64_t H, int N, int dk, bool bf16,
                                 cudaStream_t s) {
  const int smem = (2 * N * dk + 3 * N * N + 2 * N) * 4;
  if (bf16) {
    auto kern = attention_map_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(B * H), kDiagThreads, smem, s>>>(static_cast<const __nv_bfloat16 *>(q),
                                                       static_cast<const __nv_bfloat16 *>(k), beta,
                                                       g, attn, (int)H, N, dk);
  } else {
    auto kern = attention_map_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(B * H), kDiagThreads, smem, s>>>(static_cast<const float *>(q),
                                                       static_cast<const float *>(k), beta, g,
                                                       attn, (int)H, N, dk);
  }
  return cudaGetLastError();
}

}  // namespace delta
